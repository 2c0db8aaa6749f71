// Allocation-free entry point: smla_l1norm_run_noalloc().
//
// Who needs it: callers that cannot call cudaMalloc -- code running where a
// framework's caching allocator owns all device memory, plugins that are
// handed device pointers but no allocator, or deployments that forbid
// allocation after start-up.  The plan-based path allocates its work list
// and status word in smla_l1norm_plan_create(); this variant keeps both in a
// fixed, file-scope device array instead, so a call needs only the caller's
// inputs and outputs.
//
// The scratch array is static device memory: every GPU that loads this
// library holds kScratchBytes of it until the process exits.  All calls on a
// device share it and it keeps the last call's contents; each call rewrites
// the work list and clears the status word before its kernel runs.  Calls
// that overlap on the GPU (different streams, or the same plan-less call
// issued concurrently from several host threads onto different streams)
// race on the array and must be avoided.
//
// In host code the array's name is only a host-side stand-in for the device
// symbol, never a device address: the real address is fetched once per
// device with cudaGetSymbolAddress (with that device current) and cached.
// That set-up happens in the first call on each device, so the first call on
// a device should come before any stream capture.
//
// No device memory is allocated and no host heap memory either: the work
// list is built in fixed host staging arrays (guarded by a mutex) and copied
// into the device array with one cudaMemcpyAsync.  The article
// ("SparseFlashMlaSoftmaxL1Norm", CANN ops-transformer) has no counterpart of
// this entry point; the operator it runs is the same fused kernel.

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/smla_l1norm.h"
#include "smla_internal.h"

namespace {

using smla::WorkItem;

constexpr int kMaxCtas = 1024;
constexpr int kMaxItems = 65536;
constexpr size_t kStatusBytes = 256;
constexpr size_t kOffsetsBytes = ((sizeof(int32_t) * (kMaxCtas + 1) + 255) / 256) * 256;
constexpr size_t kScratchBytes = kStatusBytes + kOffsetsBytes + sizeof(WorkItem) * kMaxItems;
constexpr int kMaxDevices = 64;

// The scratch: [status word | CTA offsets | work items].
static __device__ __align__(256) uint8_t g_smla_scratch[kScratchBytes];

std::mutex g_mutex;                       // guards everything below
void* g_scratch_dev[kMaxDevices] = {};    // device address of g_smla_scratch, per device
// Host staging: the bytes copied to the scratch, and the items in token order.
alignas(256) uint8_t g_stage[kScratchBytes];
WorkItem g_items_in_order[kMaxItems];

smla_status fail_cuda(cudaError_t) { return SMLA_ERR_CUDA; }

struct Shape {
  bool sparse, tnd;
  int G, R, n_mma, width, batch;
  int64_t n_tokens, q_rows, k_rows, n_items;
};

int64_t seq_len(const int32_t* cu, int b) { return static_cast<int64_t>(cu[b + 1]) - cu[b]; }

// The same checks as smla_l1norm_plan_create, without building anything.
smla_status check_desc(const smla_l1norm_desc* d, Shape* s) {
  if (d == nullptr) return SMLA_ERR_NULLPTR;
  if (d->layout_q != SMLA_LAYOUT_BSND && d->layout_q != SMLA_LAYOUT_TND) return SMLA_ERR_INVALID;
  if (d->layout_k != d->layout_q) return SMLA_ERR_INVALID;
  if (d->dtype != SMLA_DTYPE_F16 && d->dtype != SMLA_DTYPE_BF16) return SMLA_ERR_INVALID;
  if (d->num_heads_k != 1) return SMLA_ERR_INVALID;
  if (d->num_heads_q < 1 || d->num_heads_q > 128) return SMLA_ERR_INVALID;
  if (d->head_dim != smla::kHeadDim) return SMLA_ERR_INVALID;
  if (d->mask_mode == 1 || d->mask_mode == 2) return SMLA_ERR_UNSUPPORTED;
  if (d->mask_mode != 0 && d->mask_mode != 3) return SMLA_ERR_INVALID;
  if (d->cmp_ratio < 1 || d->cmp_ratio > 128) return SMLA_ERR_INVALID;
  if (d->cmp_ratio != 1) return SMLA_ERR_UNSUPPORTED;
  if (d->topk < 0) return SMLA_ERR_INVALID;
  if (!std::isfinite(d->softmax_scale)) return SMLA_ERR_INVALID;
  if (d->has_topk_length != 0 && d->has_topk_length != 1) return SMLA_ERR_INVALID;
  if (d->has_topk_length && d->topk == 0) return SMLA_ERR_INVALID;
  if (d->num_ctas < 0) return SMLA_ERR_INVALID;
  if (d->topk_length_hint != nullptr && d->topk == 0) return SMLA_ERR_INVALID;
  s->sparse = d->topk > 0;
  s->tnd = d->layout_q == SMLA_LAYOUT_TND;
  s->G = d->num_heads_q;
  s->R = s->sparse ? 1 : std::max(1, 128 / s->G);
  s->n_mma = static_cast<int>(std::max<int64_t>(16, ((static_cast<int64_t>(s->R) * s->G + 15) / 16) * 16));
  s->batch = d->batch_size;
  if (d->batch_size < 0) return SMLA_ERR_INVALID;
  s->n_items = 0;
  if (s->tnd) {
    if (d->cu_seqlens_q == nullptr || d->cu_seqlens_k == nullptr) return SMLA_ERR_NULLPTR;
    if (d->cu_seqlens_q[0] != 0 || d->cu_seqlens_k[0] != 0) return SMLA_ERR_INVALID;
    int64_t max_sk = 0;
    for (int b = 0; b < s->batch; ++b) {
      if (seq_len(d->cu_seqlens_q, b) < 0 || seq_len(d->cu_seqlens_k, b) < 0) return SMLA_ERR_INVALID;
      max_sk = std::max(max_sk, seq_len(d->cu_seqlens_k, b));
      s->n_items += s->sparse ? seq_len(d->cu_seqlens_q, b) : (seq_len(d->cu_seqlens_q, b) + s->R - 1) / s->R;
    }
    s->n_tokens = d->cu_seqlens_q[s->batch];
    s->k_rows = d->cu_seqlens_k[s->batch];
    if (!s->sparse && d->max_seqlen_k < max_sk) return SMLA_ERR_INVALID;
    s->width = s->sparse ? d->topk : d->max_seqlen_k;
  } else {
    if (d->max_seqlen_q < 0 || d->max_seqlen_k < 0) return SMLA_ERR_INVALID;
    s->n_tokens = static_cast<int64_t>(s->batch) * d->max_seqlen_q;
    s->k_rows = static_cast<int64_t>(s->batch) * d->max_seqlen_k;
    s->n_items = s->sparse ? s->n_tokens
                           : static_cast<int64_t>(s->batch) * ((d->max_seqlen_q + s->R - 1) / s->R);
    s->width = s->sparse ? d->topk : d->max_seqlen_k;
  }
  s->q_rows = s->n_tokens * s->G;
  if (s->q_rows + 256 >= (int64_t{1} << 31) || s->k_rows + 256 >= (int64_t{1} << 31)) return SMLA_ERR_INVALID;
  if (s->n_tokens * static_cast<int64_t>(s->width) >= (int64_t{1} << 40)) return SMLA_ERR_INVALID;
  return SMLA_OK;
}

int visible(int64_t r, int64_t Sq, int64_t Sk, int mask_mode) {
  if (mask_mode == 0) return static_cast<int>(Sk);
  return static_cast<int>(std::min<int64_t>(Sk, std::max<int64_t>(0, r + Sk - Sq + 1)));
}

// Work items in token order into g_items_in_order (same fields as the
// plan-based schedule).
void fill_items(const smla_l1norm_desc* d, const Shape& s) {
  int64_t n = 0;
  for (int b = 0; b < s.batch; ++b) {
    const int64_t q0 = s.tnd ? d->cu_seqlens_q[b] : static_cast<int64_t>(b) * d->max_seqlen_q;
    const int64_t k0 = s.tnd ? d->cu_seqlens_k[b] : static_cast<int64_t>(b) * d->max_seqlen_k;
    const int64_t Sq = s.tnd ? seq_len(d->cu_seqlens_q, b) : d->max_seqlen_q;
    const int64_t Sk = s.tnd ? seq_len(d->cu_seqlens_k, b) : d->max_seqlen_k;
    for (int64_t r0 = 0; r0 < Sq; r0 += s.R) {
      const int64_t nrows = std::min<int64_t>(s.R, Sq - r0);
      int64_t tiles = 0;
      if (!s.sparse) {
        const int64_t vis = visible(r0 + nrows - 1, Sq, Sk, d->mask_mode);
        tiles = (std::min<int64_t>(vis, s.width) + smla::kTileKeys - 1) / smla::kTileKeys;
      }
      g_items_in_order[n++] = WorkItem{static_cast<int32_t>(q0 + r0), static_cast<int32_t>(nrows),
                                       static_cast<int32_t>(r0), static_cast<int32_t>(k0),
                                       static_cast<int32_t>(Sq), static_cast<int32_t>(Sk),
                                       static_cast<int32_t>(tiles), b};
    }
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_rows(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows, int dtype) {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(smla::kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(smla::kHeadDim) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(smla::kChunkElems), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == SMLA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" smla_status smla_l1norm_run_noalloc(const smla_l1norm_desc* desc, const void* q, const void* k,
                                               const float* softmax_lse, const int32_t* sparse_indices,
                                               const int32_t* topk_length, float* out, smla_stream_t stream) {
  Shape s;
  smla_status st = check_desc(desc, &s);
  if (st != SMLA_OK) return st;
  if (s.n_items > kMaxItems) return SMLA_ERR_CAPACITY;  // the fixed scratch holds kMaxItems items
  if (s.n_tokens == 0 || s.width == 0) return SMLA_OK;
  if (q == nullptr || softmax_lse == nullptr || out == nullptr) return SMLA_ERR_NULLPTR;
  if (s.k_rows > 0 && k == nullptr) return SMLA_ERR_NULLPTR;
  if (s.sparse && sparse_indices == nullptr) return SMLA_ERR_NULLPTR;
  if (desc->has_topk_length && topk_length == nullptr) return SMLA_ERR_NULLPTR;
  if (!al16(q) || (k != nullptr && !al16(k)) || !al4(softmax_lse) || !al4(out) ||
      (sparse_indices != nullptr && !al4(sparse_indices)) || (topk_length != nullptr && !al4(topk_length)))
    return SMLA_ERR_INVALID;

  std::lock_guard<std::mutex> lock(g_mutex);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_CAPACITY;
  if (g_scratch_dev[dev] == nullptr) {
    // one-time set-up on this device: the device address of the scratch array
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_smla_scratch);
    if (e != cudaSuccess || ptr == nullptr) return fail_cuda(e);
    g_scratch_dev[dev] = ptr;
  }
  int sms = 0, optin = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  int ctas = desc->num_ctas > 0 ? desc->num_ctas : sms;
  ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({static_cast<int64_t>(ctas), s.n_items,
                                                                   static_cast<int64_t>(kMaxCtas)})));
  int stages = smla::kMaxStages;
  while (stages > 2 && smla::smem_bytes_for(s.n_mma, stages) > optin) --stages;
  const int smem = smla::smem_bytes_for(s.n_mma, stages);
  if (smem > optin) return SMLA_ERR_INVALID;

  // Work list: items dealt to CTAs in a stride over the tokens taken in
  // reverse order (late causal rows see the most keys, so this spreads the
  // heavy rows evenly); each CTA's items are contiguous, as the kernel reads them.
  fill_items(desc, s);
  std::memset(g_stage, 0, kStatusBytes);  // status word starts at zero
  auto* offs = reinterpret_cast<int32_t*>(g_stage + kStatusBytes);
  auto* items = reinterpret_cast<WorkItem*>(g_stage + kStatusBytes + kOffsetsBytes);
  int64_t pos = 0;
  for (int c = 0; c < ctas; ++c) {
    offs[c] = static_cast<int32_t>(pos);
    for (int64_t i = c; i < s.n_items; i += ctas) items[pos++] = g_items_in_order[s.n_items - 1 - i];
  }
  offs[ctas] = static_cast<int32_t>(pos);
  uint8_t* dbase = static_cast<uint8_t*>(g_scratch_dev[dev]);
  auto cstream = reinterpret_cast<cudaStream_t>(stream);
  // pageable source: the copy has taken the bytes when the call returns, and
  // it is ordered after earlier work on this stream
  e = cudaMemcpyAsync(dbase, g_stage, kStatusBytes + sizeof(int32_t) * (ctas + 1), cudaMemcpyHostToDevice, cstream);
  if (e == cudaSuccess && pos > 0)
    e = cudaMemcpyAsync(dbase + kStatusBytes + kOffsetsBytes, items, sizeof(WorkItem) * pos,
                        cudaMemcpyHostToDevice, cstream);
  if (e != cudaSuccess) return fail_cuda(e);

  CUtensorMap tq;
  const int q_box = s.R * s.G;
  if (!encode_rows(&tq, q, s.q_rows, q_box, desc->dtype)) return SMLA_ERR_CUDA;
  const int64_t mma_m = 128;
  const uint32_t ab = desc->dtype == SMLA_DTYPE_BF16 ? 1u : 0u;
  const uint32_t idesc = (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(s.n_mma >> 3) << 17) |
                         (static_cast<uint32_t>(mma_m >> 4) << 24);
  smla::KernelParams p{};
  p.k = static_cast<const uint8_t*>(k);
  p.items = reinterpret_cast<const WorkItem*>(dbase + kStatusBytes + kOffsetsBytes);
  p.cta_begin = reinterpret_cast<const int32_t*>(dbase + kStatusBytes);
  p.status = reinterpret_cast<int32_t*>(dbase);
  p.lse = softmax_lse;
  p.idx = s.sparse ? sparse_indices : nullptr;
  p.topk_len = desc->has_topk_length ? topk_length : nullptr;
  p.out = out;
  p.G = s.G;
  p.R = s.R;
  p.n_mma = s.n_mma;
  p.q_box_rows = q_box;
  p.topk = s.sparse ? desc->topk : 0;
  p.width = s.width;
  p.mask_mode = desc->mask_mode;
  p.stages = stages;
  p.idesc = static_cast<int32_t>(idesc);
  p.c_log2 = static_cast<float>(static_cast<double>(desc->softmax_scale) * 1.4426950408889634);
  p.inv_g = 1.0f / static_cast<float>(s.G);
  p.timeout_ns = 2000LL * 1000000LL;
  e = smla::configure_fused(smem);
  if (e == cudaSuccess) e = smla::launch_fused(p, tq, s.sparse, smla::kModeL1, ctas, smem, cstream);
  if (e != cudaSuccess) return fail_cuda(e);
  return SMLA_OK;
}
