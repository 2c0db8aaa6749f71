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
// into the device array with cudaMemcpyAsync.  Validation, the key-ring depth
// rule, the instruction descriptor, the tensor-map encoding and the wait
// limit are the plan path's own functions (smla_internal.h), so the two
// entry points cannot drift apart.  The article
// ("SparseFlashMlaSoftmaxL1Norm", CANN ops-transformer) has no counterpart of
// this entry point; the operator it runs is the same fused kernel.

#include <algorithm>
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

int64_t seq_len(const int32_t* cu, int b) { return static_cast<int64_t>(cu[b + 1]) - cu[b]; }

// Launch shape of one call: the same key-ring rule as a plan (even depth,
// at least kMinStages, the deepest that fits), one CTA per SM by default.
struct LaunchShape {
  int ctas, stages, smem;
};

smla_status launch_shape(const smla_l1norm_desc* d, const smla::Shape& s, int sms, int optin, LaunchShape* ls) {
  if (s.n_items > kMaxItems) return SMLA_ERR_CAPACITY;  // the fixed scratch holds kMaxItems items
  int ctas = d->num_ctas > 0 ? d->num_ctas : sms;
  ls->ctas = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>({static_cast<int64_t>(ctas), s.n_items, static_cast<int64_t>(kMaxCtas)})));
  ls->stages = smla::stages_for(s.n_mma, optin);
  ls->smem = smla::smem_bytes_for(s.n_mma, ls->stages);
  if (ls->smem > optin) return SMLA_ERR_INVALID;
  return SMLA_OK;
}

// Work items in token order into g_items_in_order (the fields the plan-based
// schedule gives them).
void fill_items(const smla_l1norm_desc* d, const smla::Shape& s) {
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
        const int64_t vis = smla::visible_keys(r0 + nrows - 1, Sq, Sk, d->mask_mode, d->cmp_ratio);
        tiles = (std::min<int64_t>(vis, s.width) + smla::kTileKeys - 1) / smla::kTileKeys;
      }
      g_items_in_order[n++] = WorkItem{static_cast<int32_t>(q0 + r0), static_cast<int32_t>(nrows),
                                       static_cast<int32_t>(r0), static_cast<int32_t>(k0),
                                       static_cast<int32_t>(Sq), static_cast<int32_t>(Sk),
                                       static_cast<int32_t>(tiles), b};
    }
  }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" smla_status smla_debug_noalloc_config(const smla_l1norm_desc* desc, int32_t num_sms, int32_t smem_optin,
                                                 smla_plan_info* info) {
  if (info == nullptr) return SMLA_ERR_NULLPTR;
  if (num_sms <= 0 || smem_optin <= 0) return SMLA_ERR_INVALID;
  smla::Shape s;
  smla_status st = smla::check_desc(desc, &s);
  if (st != SMLA_OK) return st;
  LaunchShape ls;
  st = launch_shape(desc, s, num_sms, smem_optin, &ls);
  if (st != SMLA_OK) return st;
  std::memset(info, 0, sizeof(*info));
  info->num_tokens = s.n_tokens;
  info->num_items = s.n_items;
  info->num_ctas = ls.ctas;
  info->rows_per_item = s.R;
  info->mma_n = s.n_mma;
  info->stages = ls.stages;
  info->smem_bytes = ls.smem;
  info->out_width = s.width;
  info->q_rows_total = s.q_rows;
  info->k_rows_total = s.k_rows;
  info->mma_issuers = smla::l1_issuers(s);
  return SMLA_OK;
}

extern "C" smla_status smla_l1norm_run_noalloc(const smla_l1norm_desc* desc, const void* q, const void* k,
                                               const float* softmax_lse, const int32_t* sparse_indices,
                                               const int32_t* topk_length, float* out, smla_stream_t stream) {
  smla::Shape s;
  smla_status st = smla::check_desc(desc, &s);
  if (st != SMLA_OK) return st;
  // compressed keys under the causal mask need cmp_residual_k, which this
  // entry point has no argument for
  if (desc->cmp_ratio != 1 && desc->mask_mode == 3) return SMLA_ERR_UNSUPPORTED;
  if (s.n_items > kMaxItems) return SMLA_ERR_CAPACITY;  // before any CUDA call
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
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_CAPACITY;
  if (g_scratch_dev[dev] == nullptr) {
    // one-time set-up on this device: the device address of the scratch array
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_smla_scratch);
    if (e != cudaSuccess || ptr == nullptr) return SMLA_ERR_CUDA;
    g_scratch_dev[dev] = ptr;
  }
  int sms = 0, optin = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  LaunchShape ls;
  st = launch_shape(desc, s, sms, optin, &ls);
  if (st != SMLA_OK) return st;

  // Work list: items dealt to CTAs in a stride over the tokens taken in
  // reverse order (late causal rows see the most keys, so this spreads the
  // heavy rows evenly); each CTA's items are contiguous, as the kernel reads them.
  fill_items(desc, s);
  std::memset(g_stage, 0, kStatusBytes);  // status word starts at zero
  auto* offs = reinterpret_cast<int32_t*>(g_stage + kStatusBytes);
  auto* items = reinterpret_cast<WorkItem*>(g_stage + kStatusBytes + kOffsetsBytes);
  int64_t pos = 0;
  for (int c = 0; c < ls.ctas; ++c) {
    offs[c] = static_cast<int32_t>(pos);
    for (int64_t i = c; i < s.n_items; i += ls.ctas) items[pos++] = g_items_in_order[s.n_items - 1 - i];
  }
  offs[ls.ctas] = static_cast<int32_t>(pos);
  uint8_t* dbase = static_cast<uint8_t*>(g_scratch_dev[dev]);
  auto cstream = reinterpret_cast<cudaStream_t>(stream);
  // Pageable source: cudaMemcpyAsync stages the host bytes before it
  // returns, and the device copy is ordered after earlier work on ``stream``.
  e = cudaMemcpyAsync(dbase, g_stage, kStatusBytes + sizeof(int32_t) * (ls.ctas + 1), cudaMemcpyHostToDevice,
                      cstream);
  if (e == cudaSuccess && pos > 0)
    e = cudaMemcpyAsync(dbase + kStatusBytes + kOffsetsBytes, items, sizeof(WorkItem) * pos,
                        cudaMemcpyHostToDevice, cstream);
  if (e != cudaSuccess) return SMLA_ERR_CUDA;

  CUtensorMap tq;
  const int q_box = s.R * s.G;
  if (!smla::encode_rows_map(&tq, q, s.q_rows, q_box, desc->dtype)) return SMLA_ERR_CUDA;
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
  p.cmp_ratio = desc->cmp_ratio;
  p.stages = ls.stages;
  p.idesc = static_cast<int32_t>(smla::make_idesc(desc->dtype, s.n_mma));
  p.idesc_lse = static_cast<int32_t>(smla::make_idesc(desc->dtype, smla::kTileKeys));
  p.c_log2 = static_cast<float>(static_cast<double>(desc->softmax_scale) * 1.4426950408889634);
  p.inv_g = 1.0f / static_cast<float>(s.G);
  p.timeout_ns = smla::wait_timeout_ns();
  e = smla::configure_fused_for_device();
  if (e == cudaSuccess)
    e = smla::launch_fused(p, tq, s.sparse, smla::kModeL1, smla::l1_issuers(s), ls.ctas, ls.smem, cstream);
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}
