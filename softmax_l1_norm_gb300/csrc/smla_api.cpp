// Host side of the C ABI declared in include/smla_l1norm.h: validation,
// the CTA work schedule (the GB300 counterpart of the article's metadata
// operator), tensor-map encoding and the launch.
//
// Validation follows the article "SparseFlashMlaSoftmaxL1Norm" (CANN
// ops-transformer): parameter tables (参数说明), constraints (约束说明) and the
// aclnn error split between null pointers and invalid parameters.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <queue>
#include <string>
#include <vector>

#include "../../include/smla_l1norm.h"
#include "smla_internal.h"

namespace smla {
cudaError_t launch_wait_timeout_probe(int32_t* status, int64_t timeout_ns, cudaStream_t stream);
}

using smla::WorkItem;

namespace {

thread_local std::string g_last_cuda_error;

smla_status cuda_fail(cudaError_t e, const char* what) {
  g_last_cuda_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return SMLA_ERR_CUDA;
}

constexpr int kDefaultSmemOptin = 232448;  // 227 KB, the sm_100-family opt-in limit

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// A validated description plus its per-sequence offsets and lengths.
struct Geometry : smla::Shape {
  std::vector<int64_t> q0, sq, k0, sk;  // per sequence
};

smla_status validate(const smla_l1norm_desc* d, Geometry* g) {
  smla_status st = smla::check_desc(d, g);
  if (st != SMLA_OK) return st;
  for (int b = 0; b < g->batch; ++b) {
    if (g->tnd) {
      g->q0.push_back(d->cu_seqlens_q[b]);
      g->sq.push_back(static_cast<int64_t>(d->cu_seqlens_q[b + 1]) - d->cu_seqlens_q[b]);
      g->k0.push_back(d->cu_seqlens_k[b]);
      g->sk.push_back(static_cast<int64_t>(d->cu_seqlens_k[b + 1]) - d->cu_seqlens_k[b]);
    } else {
      g->q0.push_back(static_cast<int64_t>(b) * d->max_seqlen_q);
      g->sq.push_back(d->max_seqlen_q);
      g->k0.push_back(static_cast<int64_t>(b) * d->max_seqlen_k);
      g->sk.push_back(d->max_seqlen_k);
    }
  }
  return SMLA_OK;
}

}  // namespace

namespace smla {

// Checks every field of the description ([SMLA] 参数说明 and 约束说明) and
// derives the launch geometry.  Reads the host cu_seqlens arrays in TND.
smla_status check_desc(const smla_l1norm_desc* d, Shape* g) {
  if (d == nullptr) return SMLA_ERR_NULLPTR;
  if (d->layout_q != SMLA_LAYOUT_BSND && d->layout_q != SMLA_LAYOUT_TND) return SMLA_ERR_INVALID;
  if (d->layout_k != d->layout_q) return SMLA_ERR_INVALID;  // layout_q must equal layout_k
  if (d->dtype != SMLA_DTYPE_F16 && d->dtype != SMLA_DTYPE_BF16) return SMLA_ERR_INVALID;
  if (d->num_heads_k != 1) return SMLA_ERR_INVALID;                          // N2 only 1
  if (d->num_heads_q < 1 || d->num_heads_q > 128) return SMLA_ERR_INVALID;   // N1 in 1..128
  if (d->num_heads_q % d->num_heads_k != 0) return SMLA_ERR_INVALID;
  if (d->head_dim != kHeadDim) return SMLA_ERR_INVALID;                      // D only 512
  if (d->mask_mode == 1 || d->mask_mode == 2) return SMLA_ERR_UNSUPPORTED;
  if (d->mask_mode != 0 && d->mask_mode != 3) return SMLA_ERR_INVALID;
  if (d->cmp_ratio < 1 || d->cmp_ratio > 128) return SMLA_ERR_INVALID;       // range 1..128
  if (d->topk < 0) return SMLA_ERR_INVALID;
  if (!std::isfinite(d->softmax_scale)) return SMLA_ERR_INVALID;
  if (d->has_topk_length != 0 && d->has_topk_length != 1) return SMLA_ERR_INVALID;
  if (d->has_topk_length && d->topk == 0) return SMLA_ERR_INVALID;  // topk_length needs indices
  if (d->num_ctas < 0) return SMLA_ERR_INVALID;

  *g = Shape{};
  g->sparse = d->topk > 0;
  g->tnd = d->layout_q == SMLA_LAYOUT_TND;
  g->G = d->num_heads_q / d->num_heads_k;
  g->R = g->sparse ? 1 : std::max(1, 128 / g->G);
  g->n_mma = static_cast<int>(std::max<int64_t>(16, ceil_div(static_cast<int64_t>(g->R) * g->G, 16) * 16));
  if (g->tnd) {
    if (d->cu_seqlens_q == nullptr || d->cu_seqlens_k == nullptr) return SMLA_ERR_NULLPTR;
    if (d->batch_size < 0) return SMLA_ERR_INVALID;
    g->batch = d->batch_size;
    const int32_t* cq = d->cu_seqlens_q;
    const int32_t* ck = d->cu_seqlens_k;
    if (cq[0] != 0 || ck[0] != 0) return SMLA_ERR_INVALID;
    int64_t max_sk = 0;
    for (int b = 0; b < g->batch; ++b) {
      if (cq[b + 1] < cq[b] || ck[b + 1] < ck[b]) return SMLA_ERR_INVALID;
      const int64_t sq = static_cast<int64_t>(cq[b + 1]) - cq[b];
      max_sk = std::max<int64_t>(max_sk, static_cast<int64_t>(ck[b + 1]) - ck[b]);
      g->n_items += g->sparse ? sq : ceil_div(sq, g->R);
    }
    g->n_tokens = cq[g->batch];
    g->k_rows = ck[g->batch];
    if (g->sparse) {
      g->width = d->topk;
    } else {
      if (d->max_seqlen_k < max_sk) return SMLA_ERR_INVALID;  // output width must hold every row
      g->width = d->max_seqlen_k;
    }
  } else {
    if (d->batch_size < 0 || d->max_seqlen_q < 0 || d->max_seqlen_k < 0) return SMLA_ERR_INVALID;
    g->batch = d->batch_size;
    g->n_tokens = static_cast<int64_t>(g->batch) * d->max_seqlen_q;
    g->k_rows = static_cast<int64_t>(g->batch) * d->max_seqlen_k;
    g->width = g->sparse ? d->topk : d->max_seqlen_k;
    g->n_items = g->sparse ? g->n_tokens : static_cast<int64_t>(g->batch) * ceil_div(d->max_seqlen_q, g->R);
  }
  g->q_rows = g->n_tokens * g->G;
  // TMA coordinates are 32-bit; keep every row index representable.
  if (g->q_rows + 256 >= (int64_t{1} << 31) || g->k_rows + 256 >= (int64_t{1} << 31)) return SMLA_ERR_INVALID;
  if (g->n_tokens * static_cast<int64_t>(g->width) >= (int64_t{1} << 40)) return SMLA_ERR_INVALID;
  if (d->topk_length_hint != nullptr && !g->sparse) return SMLA_ERR_INVALID;
  return SMLA_OK;
}

int visible_keys(int64_t r, int64_t Sq, int64_t Sk, int mask_mode, int cmp_ratio) {
  if (mask_mode == 0) return static_cast<int>(Sk);
  const int64_t c = std::max(1, cmp_ratio);
  const int64_t d = r + Sk * c + (c - 1) - Sq + 1;  // the largest residual, c - 1
  return static_cast<int>(std::min<int64_t>(Sk, std::max<int64_t>(0, d) / c));
}

}  // namespace smla

namespace {

using smla::visible_keys;

struct Schedule {
  std::vector<WorkItem> items;       // grouped by CTA
  std::vector<int32_t> cta_begin;    // num_ctas + 1
  int64_t est_tiles = 0;
  double max_cost = 0, mean_cost = 0;
};

// Build the work items and deal them to CTAs by longest-processing-time
// first: items sorted by estimated cost, each given to the least-loaded CTA.
// Any assignment gives the same output bits; the schedule only balances
// time.  Cost of an item: its 128-key tiles, plus a per-token overhead for
// the q load and the zero tail.
Schedule build_schedule(const smla_l1norm_desc* d, const Geometry& g, int num_ctas, int64_t tok_lo = 0,
                        int64_t tok_hi = INT64_MAX, bool pair = false, int64_t split = 0) {
  Schedule s;
  std::vector<WorkItem> items;
  std::vector<double> cost;
  const double row_overhead = 0.05 + 0.35 * (g.n_mma / 128.0);
  for (int b = 0; b < g.batch; ++b) {
    const int64_t Sq = g.sq[b], Sk = g.sk[b];
    if (g.sparse) {
      for (int64_t r = 0; r < Sq; ++r) {
        const int64_t tok = g.q0[b] + r;
        if (tok < tok_lo || tok >= tok_hi) continue;
        int64_t n;
        if (d->topk_length_hint != nullptr) {
          n = std::min<int64_t>(std::max<int32_t>(d->topk_length_hint[tok], 0), d->topk);
        } else if (d->has_topk_length) {
          n = std::min<int64_t>(d->topk, visible_keys(r, Sq, Sk, d->mask_mode, d->cmp_ratio));
        } else {
          n = d->topk;
        }
        if (Sk == 0) n = 0;
        const int64_t tiles = ceil_div(n, smla::kTileKeys);
        WorkItem w{static_cast<int32_t>(tok), 1, static_cast<int32_t>(r), static_cast<int32_t>(g.k0[b]),
                   static_cast<int32_t>(Sq), static_cast<int32_t>(Sk), 0, b};
        items.push_back(w);
        // a CTA pair runs two tiles per step
        cost.push_back(static_cast<double>(pair ? ceil_div(tiles, 2) : tiles) + row_overhead +
                       0.02 * static_cast<double>(g.width - tiles * smla::kTileKeys) / smla::kTileKeys);
        s.est_tiles += tiles;
      }
    } else {
      for (int64_t r0 = 0; r0 < Sq; r0 += g.R) {
        if (g.q0[b] + r0 < tok_lo || g.q0[b] + r0 >= tok_hi) continue;
        const int64_t nrows = std::min<int64_t>(g.R, Sq - r0);
        const int64_t vis = visible_keys(r0 + nrows - 1, Sq, Sk, d->mask_mode, d->cmp_ratio);
        const int64_t tiles = ceil_div(std::min<int64_t>(vis, g.width), smla::kTileKeys);
        // one item, or (split > 0) as few parts of at most `split` key tiles
        // as cover the pack, of equal size to within one tile; the last part
        // (or the only one) zeroes the rest of the rows
        const int64_t nparts = split > 0 ? std::max<int64_t>(1, ceil_div(tiles, split)) : 1;
        const int64_t part = std::max<int64_t>(1, ceil_div(tiles, nparts));
        for (int64_t t0 = 0; t0 == 0 || t0 < tiles; t0 += part) {
          const int64_t n = std::min<int64_t>(part, tiles - t0);
          const bool last = t0 + part >= tiles;
          WorkItem w{static_cast<int32_t>(g.q0[b] + r0), static_cast<int32_t>(nrows), static_cast<int32_t>(r0),
                     static_cast<int32_t>(g.k0[b]), static_cast<int32_t>(Sq), static_cast<int32_t>(Sk),
                     static_cast<int32_t>(std::max<int64_t>(n, 0)), b};
          w.t0 = static_cast<int32_t>(t0);
          w.cut_tail = last ? 0 : 1;
          items.push_back(w);
          const double tail = last ? static_cast<double>(g.width - tiles * smla::kTileKeys) / smla::kTileKeys : 0.0;
          cost.push_back(static_cast<double>(std::max<int64_t>(n, 0)) + row_overhead + 0.02 * nrows * tail);
        }
        s.est_tiles += tiles;
      }
    }
  }
  const int64_t n = static_cast<int64_t>(items.size());
  std::vector<int64_t> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return cost[a] > cost[b]; });
  using Load = std::pair<double, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < num_ctas; ++c) heap.push({0.0, c});
  std::vector<std::vector<int64_t>> per(num_ctas);
  std::vector<double> load(num_ctas, 0.0);
  for (int64_t i : order) {
    Load l = heap.top();
    heap.pop();
    per[l.second].push_back(i);
    l.first += cost[i];
    load[l.second] = l.first;
    heap.push(l);
  }
  s.cta_begin.resize(num_ctas + 1);
  s.items.reserve(n);
  for (int c = 0; c < num_ctas; ++c) {
    s.cta_begin[c] = static_cast<int32_t>(s.items.size());
    // within a CTA, keep token order (neighbouring tokens share keys in L2)
    std::sort(per[c].begin(), per[c].end());
    for (int64_t i : per[c]) s.items.push_back(items[i]);
  }
  s.cta_begin[num_ctas] = static_cast<int32_t>(s.items.size());
  if (num_ctas > 0) {
    s.max_cost = *std::max_element(load.begin(), load.end());
    s.mean_cost = std::accumulate(load.begin(), load.end(), 0.0) / num_ctas;
  }
  return s;
}

// Dense form: when a few long token packs would leave most CTAs waiting for
// the heaviest (few packs, many key tiles each), the L1-norm launch splits
// each pack's key tiles into parts of at most `split` tiles, which the
// scheduler deals out separately; a part reloads its pack's q block.  The
// part size chosen is the one whose schedule has the lightest heaviest CTA,
// kept when it beats the unsplit schedule `base` by at least 10 %; 0 = no
// split.  `force` (the SMLA_SPLIT variable, may be null) fixes the part size
// (0: no split).  The forward-LSE launches reduce over a row's keys and always
// take whole packs.
int64_t choose_split(const smla_l1norm_desc* d, const Geometry& g, int num_ctas, const Schedule& base,
                     const char* force) {
  if (g.sparse) return 0;
  int64_t max_tiles = 0;
  for (const WorkItem& w : base.items) max_tiles = std::max<int64_t>(max_tiles, w.ntiles);
  int64_t best = 0;
  if (force != nullptr) {
    best = std::max<int64_t>(0, std::atoll(force));
  } else if (max_tiles > 1 && static_cast<int64_t>(base.items.size()) < 8 * static_cast<int64_t>(num_ctas)) {
    double best_cost = 0.9 * base.max_cost;
    for (int64_t cap = 1; cap < max_tiles; cap = cap < 4 ? cap + 1 : cap * 2) {
      const Schedule t = build_schedule(d, g, num_ctas, 0, INT64_MAX, false, cap);
      if (t.max_cost < best_cost) {
        best_cost = t.max_cost;
        best = cap;
      }
    }
  }
  return (best > 0 && best < max_tiles) ? best : 0;
}

void fill_info(const Geometry& g, const Schedule& s, int num_ctas, int stages, int smem, smla_plan_info* info) {
  std::memset(info, 0, sizeof(*info));
  info->num_tokens = g.n_tokens;
  info->num_items = static_cast<int64_t>(s.items.size());
  info->num_ctas = num_ctas;
  info->rows_per_item = g.R;
  info->mma_n = g.n_mma;
  info->stages = stages;
  info->smem_bytes = smem;
  info->out_width = g.width;
  info->est_tiles = s.est_tiles;
  info->max_cta_cost = s.max_cost;
  info->mean_cta_cost = s.mean_cost;
  info->q_rows_total = g.q_rows;
  info->k_rows_total = g.k_rows;
  info->mma_issuers = smla::l1_issuers(g);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

namespace smla {

int stages_for(int n_mma, int smem_limit) {
  int st = kMaxStages;
  while (st > kMinStages && smem_bytes_for(n_mma, st) > smem_limit) st -= 2;
  return st;
}

uint32_t make_idesc(int dtype, int n_mma, int m) {
  // tcgen05 instruction descriptor, kind::f16: fp32 accumulator, A and B of
  // the same 16-bit type, both K-major, M = m, N = n_mma.
  const uint32_t ab = dtype == SMLA_DTYPE_BF16 ? 1u : 0u;
  uint32_t d = 0;
  d |= 1u << 4;                                    // D format: f32
  d |= ab << 7;                                    // A format
  d |= ab << 10;                                   // B format
  d |= static_cast<uint32_t>(n_mma >> 3) << 17;    // N / 8
  d |= static_cast<uint32_t>(m >> 4) << 24;        // M / 16
  return d;
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // resolved once (thread-safe static initialisation)
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

}  // namespace

// 2-D view (rows x 512) of a half-precision tensor, boxes of 64 columns x
// box_rows rows, 128-byte swizzle (the layout the MMA descriptors expect).
bool encode_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows, int dtype) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kChunkElems), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt =
      dtype == SMLA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t wait_timeout_ns() {
  if (const char* e = std::getenv("SMLA_WAIT_TIMEOUT_MS")) {
    const long long ms = std::atoll(e);
    if (ms > 0) return ms * 1000000LL;
  }
  return 2000LL * 1000000LL;  // 2 s
}

}  // namespace smla

struct smla_plan {
  smla_l1norm_desc desc;
  Geometry geo;
  int device = 0;
  int num_ctas = 0;
  int stages = 0;
  int smem = 0;
  uint32_t idesc = 0;
  void* dbuf = nullptr;
  int32_t* d_status = nullptr;
  int32_t* d_cta_begin = nullptr;
  WorkItem* d_items = nullptr;
  smla_plan_info info{};
  int64_t timeout_ns = 0;
  int32_t withhold_q = 0;            // test hook (SMLA_DEBUG_WITHHOLD_Q)
  // CTA-pair L1-norm launch (sparse, N = 128): clusters (0 = not used), its
  // ring depth and shared memory, and its own work list (one per cluster)
  int pair_clusters = 0, pair_stages = 0, pair_smem = 0;
  int32_t* d_pair_begin = nullptr;
  WorkItem* d_pair_items = nullptr;
  // Dense L1-norm launch split along the keys (0 = not split): parts of at
  // most split_tiles key tiles, with their own work list
  int split_tiles = 0;
  int32_t* d_split_begin = nullptr;
  WorkItem* d_split_items = nullptr;
  std::vector<WorkItem> items_host;  // the work list as uploaded, for the gather test hook
  // run_from_host pipeline: token chunks, each with its own work schedule,
  // so that the copies of one chunk overlap the kernel of the previous one
  std::vector<int64_t> chunk_lo, chunk_hi;
  std::vector<int32_t*> d_chunk_begin;
  std::vector<WorkItem*> d_chunk_items;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> events;  // start, end, then per chunk: inputs landed, kernel done
};

namespace {

// run_from_host pipelines over as many token chunks as leave every CTA two
// work items in each, at most kMaxHostChunks, and only when that is at least
// kMinHostChunks (else one copy, one kernel, one copy).  Measured on the
// 4096-token workload: 3.06 ms a step with 4 chunks, 3.00 with 6, 2.98 with 8.
constexpr int kMinHostChunks = 4;
constexpr int kMaxHostChunks = 8;

void release_plan(smla_plan* plan) {
  for (cudaEvent_t e : plan->events) cudaEventDestroy(e);
  if (plan->s_in != nullptr) cudaStreamDestroy(plan->s_in);
  if (plan->s_out != nullptr) cudaStreamDestroy(plan->s_out);
  if (plan->dbuf != nullptr) cudaFree(plan->dbuf);
  delete plan;
}

}  // namespace

extern "C" {

smla_status smla_l1norm_schedule_host(const smla_l1norm_desc* desc, int32_t num_ctas, int32_t split_tiles,
                                      int32_t* items, int64_t items_capacity, int32_t* cta_offsets,
                                      smla_plan_info* info) {
  Geometry g;
  smla_status st = validate(desc, &g);
  if (st != SMLA_OK) return st;
  if (num_ctas <= 0) return SMLA_ERR_INVALID;
  const Schedule base = build_schedule(desc, g, num_ctas);
  const int64_t split = split_tiles < 0 ? choose_split(desc, g, num_ctas, base, nullptr) : split_tiles;
  if (g.sparse && split > 0) return SMLA_ERR_INVALID;
  const Schedule s = split > 0 ? build_schedule(desc, g, num_ctas, 0, INT64_MAX, false, split) : base;
  if (items != nullptr) {
    const int64_t n = std::min<int64_t>(items_capacity, static_cast<int64_t>(s.items.size()));
    std::memcpy(items, s.items.data(), static_cast<size_t>(n) * sizeof(WorkItem));
  }
  if (cta_offsets != nullptr) std::memcpy(cta_offsets, s.cta_begin.data(), s.cta_begin.size() * sizeof(int32_t));
  if (info != nullptr) {
    const int stages = smla::stages_for(g.n_mma, kDefaultSmemOptin);
    fill_info(g, s, num_ctas, stages, smla::smem_bytes_for(g.n_mma, stages), info);
    info->split_tiles = static_cast<int32_t>(split);
    info->split_items = split > 0 ? static_cast<int64_t>(s.items.size()) : 0;
  }
  return SMLA_OK;
}

smla_status smla_l1norm_plan_create(const smla_l1norm_desc* desc, smla_plan** plan_out) {
  if (plan_out == nullptr) return SMLA_ERR_NULLPTR;
  *plan_out = nullptr;
  Geometry g;
  smla_status st = validate(desc, &g);
  if (st != SMLA_OK) return st;

  auto* plan = new smla_plan();
  plan->desc = *desc;
  plan->desc.cu_seqlens_q = nullptr;  // host arrays are only read here
  plan->desc.cu_seqlens_k = nullptr;
  plan->desc.topk_length_hint = nullptr;
  plan->geo = g;
  plan->idesc = smla::make_idesc(desc->dtype, g.n_mma);
  plan->timeout_ns = smla::wait_timeout_ns();
  if (const char* e = std::getenv("SMLA_DEBUG_WITHHOLD_Q")) plan->withhold_q = std::atoi(e) != 0 ? 1 : 0;

  cudaError_t e = cudaGetDevice(&plan->device);
  if (e != cudaSuccess) {
    release_plan(plan);
    return cuda_fail(e, "cudaGetDevice");
  }
  int sms = 0, optin = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, plan->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, plan->device);
  if (e != cudaSuccess) {
    release_plan(plan);
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  int ctas = desc->num_ctas > 0 ? desc->num_ctas : sms;
  ctas = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(ctas, std::max<int64_t>(1, g.n_tokens))));
  plan->num_ctas = ctas;
  plan->stages = smla::stages_for(g.n_mma, optin);
  plan->smem = smla::smem_bytes_for(g.n_mma, plan->stages);
  if (plan->smem > optin) {
    release_plan(plan);
    return SMLA_ERR_INVALID;
  }
  const Schedule s = build_schedule(desc, g, ctas);
  fill_info(g, s, ctas, plan->stages, plan->smem, &plan->info);
  plan->items_host = s.items;

  // Token chunks for run_from_host: cut the token-ordered work items into
  // runs of about equal token count (an item never straddles a cut), when
  // there is enough work for every CTA in each chunk.
  std::vector<Schedule> cs;
  const int n_chunks = static_cast<int>(
      std::min<int64_t>(kMaxHostChunks, static_cast<int64_t>(s.items.size()) / (2 * static_cast<int64_t>(ctas))));
  if (n_chunks >= kMinHostChunks) {
    std::vector<WorkItem> ordered = s.items;
    std::sort(ordered.begin(), ordered.end(), [](const WorkItem& a, const WorkItem& b) { return a.q_tok < b.q_tok; });
    int64_t cut = 0;
    plan->chunk_lo.push_back(0);
    for (const WorkItem& w : ordered) {
      const int next_chunk = static_cast<int>(plan->chunk_lo.size());
      if (next_chunk < n_chunks && w.q_tok >= g.n_tokens * next_chunk / n_chunks && w.q_tok > cut) {
        plan->chunk_hi.push_back(w.q_tok);
        plan->chunk_lo.push_back(w.q_tok);
        cut = w.q_tok;
      }
    }
    plan->chunk_hi.push_back(g.n_tokens);
    for (size_t c = 0; c < plan->chunk_lo.size(); ++c)
      cs.push_back(build_schedule(desc, g, ctas, plan->chunk_lo[c], plan->chunk_hi[c]));
  }

  // CTA pairs for the L1-norm launch (sparse form, N = 128).  The pair
  // kernel splits each token's tiles between two SMs; one MMA covers both
  // CTAs' keys and each SM holds 160 KB of keys in flight instead of 96 KB.
  // Measured on GB300 (one box, pair / single-CTA time, uniform causal and
  // clustered top-2048 selections): tokens of 4.5 tiles on average 1.06,
  // 8.5 tiles 0.99-1.01, 12.3 tiles 0.92, 14.1-15.5 tiles 0.88-0.91, from
  // 4096 to 32768 keys alike.  It runs when the schedule's mean is at least
  // kPairMinTiles tiles a token; SMLA_PAIR=0 / 1 forces the choice for
  // sparse work with exactly 128 heads.  As many clusters as fit on the
  // device at once.
  constexpr double kPairMinTiles = 10.0;
  Schedule ps;
  const char* pair_env = std::getenv("SMLA_PAIR");
  const int pair_force = pair_env == nullptr ? -1 : (std::atoi(pair_env) != 0 ? 1 : 0);
  const double mean_tiles = static_cast<double>(s.est_tiles) / static_cast<double>(std::max<int64_t>(1, g.n_tokens));
  const bool want_pair =
      pair_force == 1 || (pair_force == -1 && mean_tiles >= kPairMinTiles);
  // The pair kernel splits q into two 64-head halves and reads 128 LSE
  // entries a token: exactly 128 heads (N = 128 with no padded columns).
  if (g.sparse && g.G == 128 && g.n_mma == 128 && want_pair) {
    int clusters = 0;
    if (smla::configure_pair(optin, &clusters) == cudaSuccess && clusters > 0) {
      // a grid size the caller asked for holds for this launch too (one
      // CTA asked for: no pair)
      if (desc->num_ctas > 0) clusters = std::min(clusters, desc->num_ctas / 2);
      clusters = static_cast<int>(std::min<int64_t>(clusters, std::max<int64_t>(1, g.n_tokens)));
    } else {
      clusters = 0;
    }
    if (clusters > 0) {
      plan->pair_clusters = clusters;
      plan->pair_stages = smla::pair_stages(optin);
      plan->pair_smem = smla::pair_smem_bytes(plan->pair_stages);
      ps = build_schedule(desc, g, clusters, 0, INT64_MAX, true);
    }
    cudaGetLastError();  // a device without clusters of two: the single-CTA kernel
  }

  // Dense form: the L1-norm launch may split token packs along the keys.
  Schedule ss;
  if (!g.sparse) {
    const int64_t split = choose_split(desc, g, ctas, s, std::getenv("SMLA_SPLIT"));
    if (split > 0) {
      ss = build_schedule(desc, g, ctas, 0, INT64_MAX, false, split);
      plan->split_tiles = static_cast<int>(split);
    }
  }

  // one device buffer: status word | CTA offsets | work items | per chunk: CTA offsets | work items
  // | pair CTA offsets | pair work items | split CTA offsets | split work items
  auto round256 = [](size_t n) { return ((n + 255) / 256) * 256; };
  const size_t off_begin = 256;
  const size_t off_items = off_begin + round256(s.cta_begin.size() * sizeof(int32_t));
  size_t bytes = off_items + round256(std::max<size_t>(1, s.items.size()) * sizeof(WorkItem));
  std::vector<size_t> off_cb, off_ci;
  for (const Schedule& c : cs) {
    off_cb.push_back(bytes);
    bytes += round256(c.cta_begin.size() * sizeof(int32_t));
    off_ci.push_back(bytes);
    bytes += round256(std::max<size_t>(1, c.items.size()) * sizeof(WorkItem));
  }
  const size_t off_pb = bytes;
  bytes += round256(std::max<size_t>(1, ps.cta_begin.size()) * sizeof(int32_t));
  const size_t off_pi = bytes;
  bytes += round256(std::max<size_t>(1, ps.items.size()) * sizeof(WorkItem));
  const size_t off_sb = bytes;
  bytes += round256(std::max<size_t>(1, ss.cta_begin.size()) * sizeof(int32_t));
  const size_t off_si = bytes;
  bytes += round256(std::max<size_t>(1, ss.items.size()) * sizeof(WorkItem));
  e = cudaMalloc(&plan->dbuf, bytes);
  if (e != cudaSuccess) {
    release_plan(plan);
    return cuda_fail(e, "cudaMalloc(plan)");
  }
  std::vector<uint8_t> host(bytes, 0);
  std::memcpy(host.data() + off_begin, s.cta_begin.data(), s.cta_begin.size() * sizeof(int32_t));
  if (!s.items.empty()) std::memcpy(host.data() + off_items, s.items.data(), s.items.size() * sizeof(WorkItem));
  for (size_t c = 0; c < cs.size(); ++c) {
    std::memcpy(host.data() + off_cb[c], cs[c].cta_begin.data(), cs[c].cta_begin.size() * sizeof(int32_t));
    if (!cs[c].items.empty())
      std::memcpy(host.data() + off_ci[c], cs[c].items.data(), cs[c].items.size() * sizeof(WorkItem));
  }
  if (!ps.cta_begin.empty())
    std::memcpy(host.data() + off_pb, ps.cta_begin.data(), ps.cta_begin.size() * sizeof(int32_t));
  if (!ps.items.empty()) std::memcpy(host.data() + off_pi, ps.items.data(), ps.items.size() * sizeof(WorkItem));
  if (!ss.cta_begin.empty())
    std::memcpy(host.data() + off_sb, ss.cta_begin.data(), ss.cta_begin.size() * sizeof(int32_t));
  if (!ss.items.empty()) std::memcpy(host.data() + off_si, ss.items.data(), ss.items.size() * sizeof(WorkItem));
  e = cudaMemcpy(plan->dbuf, host.data(), bytes, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = smla::configure_fused_for_device();
  if (e == cudaSuccess && !cs.empty()) {
    e = cudaStreamCreateWithFlags(&plan->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&plan->s_out, cudaStreamNonBlocking);
    for (size_t i = 0; e == cudaSuccess && i < 2 + 2 * cs.size(); ++i) {
      cudaEvent_t ev = nullptr;
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e == cudaSuccess) plan->events.push_back(ev);
    }
  }
  if (e != cudaSuccess) {
    release_plan(plan);
    return cuda_fail(e, "plan upload");
  }
  if (plan->info.mma_issuers == 4 && !smla::four_issuers_available()) plan->info.mma_issuers = 2;
  auto* b = static_cast<uint8_t*>(plan->dbuf);
  plan->d_status = reinterpret_cast<int32_t*>(b);
  plan->d_cta_begin = reinterpret_cast<int32_t*>(b + off_begin);
  plan->d_items = reinterpret_cast<WorkItem*>(b + off_items);
  plan->d_pair_begin = reinterpret_cast<int32_t*>(b + off_pb);
  plan->d_pair_items = reinterpret_cast<WorkItem*>(b + off_pi);
  plan->info.cta_pairs = plan->pair_clusters;
  plan->d_split_begin = reinterpret_cast<int32_t*>(b + off_sb);
  plan->d_split_items = reinterpret_cast<WorkItem*>(b + off_si);
  plan->info.split_tiles = plan->split_tiles;
  plan->info.split_items = plan->split_tiles > 0 ? static_cast<int64_t>(ss.items.size()) : 0;
  plan->info.host_chunks = static_cast<int32_t>(cs.size());
  for (size_t c = 0; c < cs.size(); ++c) {
    plan->d_chunk_begin.push_back(reinterpret_cast<int32_t*>(b + off_cb[c]));
    plan->d_chunk_items.push_back(reinterpret_cast<WorkItem*>(b + off_ci[c]));
  }
  if (std::getenv("SMLA_LOG") != nullptr) {
    std::fprintf(stderr,
                 "[smla] plan: tokens=%lld items=%lld ctas=%d R=%d N=%d stages=%d smem=%d tiles=%lld "
                 "max/mean cost=%.2f/%.2f pairs=%d split=%d (max cost %.2f)\n",
                 static_cast<long long>(g.n_tokens), static_cast<long long>(s.items.size()), ctas, g.R,
                 g.n_mma, plan->stages, plan->smem, static_cast<long long>(s.est_tiles), s.max_cost,
                 s.mean_cost, plan->pair_clusters, plan->split_tiles, ss.max_cost);
  }
  *plan_out = plan;
  return SMLA_OK;
}

void smla_l1norm_plan_destroy(smla_plan* plan) {
  if (plan == nullptr) return;
  release_plan(plan);
}

smla_status smla_l1norm_output_shape(const smla_plan* plan, int64_t dims[4], int32_t* ndim) {
  if (plan == nullptr || dims == nullptr || ndim == nullptr) return SMLA_ERR_NULLPTR;
  const Geometry& g = plan->geo;
  if (g.tnd) {
    dims[0] = g.n_tokens;
    dims[1] = 1;
    dims[2] = g.width;
    dims[3] = 0;
    *ndim = 3;
  } else {
    dims[0] = g.batch;
    dims[1] = plan->desc.max_seqlen_q;
    dims[2] = 1;
    dims[3] = g.width;
    *ndim = 4;
  }
  return SMLA_OK;
}

smla_status smla_l1norm_plan_get_info(const smla_plan* plan, smla_plan_info* info) {
  if (plan == nullptr || info == nullptr) return SMLA_ERR_NULLPTR;
  *info = plan->info;
  return SMLA_OK;
}

smla_status smla_l1norm_io_sizes(const smla_plan* plan, smla_io_sizes* s) {
  if (plan == nullptr || s == nullptr) return SMLA_ERR_NULLPTR;
  const Geometry& g = plan->geo;
  s->q_bytes = static_cast<size_t>(g.q_rows) * smla::kHeadDim * 2;
  s->k_bytes = static_cast<size_t>(g.k_rows) * smla::kHeadDim * 2;
  s->lse_bytes = static_cast<size_t>(g.n_tokens) * g.G * 4;
  s->indices_bytes = g.sparse ? static_cast<size_t>(g.n_tokens) * plan->desc.topk * 4 : 0;
  s->topk_length_bytes = plan->desc.has_topk_length ? static_cast<size_t>(g.n_tokens) * 4 : 0;
  s->out_bytes = static_cast<size_t>(g.n_tokens) * g.width * 4;
  return SMLA_OK;
}

}  // extern "C"

namespace {

// Checks the tensors a mode needs and launches it.  kModeL1 reads
// t->softmax_lse and writes t->out; kModeLse writes lse_out only; kModeFused
// writes lse_out and t->out.
smla_status launch_mode(const smla_plan* plan, const smla_l1norm_tensors* t, float* lse_out, int mode,
                        smla_stream_t stream, int chunk = -1) {
  if (plan == nullptr || t == nullptr) return SMLA_ERR_NULLPTR;
  const Geometry& g = plan->geo;
  if (g.n_tokens == 0) return SMLA_OK;                       // empty q: nothing to do
  if (mode == smla::kModeL1 && g.width == 0) return SMLA_OK;  // empty output
  const bool wants_out = mode != smla::kModeLse;
  const bool wants_lse_in = mode == smla::kModeL1;
  if (t->q == nullptr) return SMLA_ERR_NULLPTR;
  if (wants_out && t->out == nullptr) return SMLA_ERR_NULLPTR;
  if (wants_lse_in && t->softmax_lse == nullptr) return SMLA_ERR_NULLPTR;
  if (!wants_lse_in && lse_out == nullptr) return SMLA_ERR_NULLPTR;
  if (g.k_rows > 0 && t->k == nullptr) return SMLA_ERR_NULLPTR;
  if (g.sparse && t->sparse_indices == nullptr) return SMLA_ERR_NULLPTR;
  if (plan->desc.has_topk_length && t->topk_length == nullptr) return SMLA_ERR_NULLPTR;
  // compressed keys with the causal mask need the per-sequence residual
  const bool needs_res = plan->desc.cmp_ratio != 1 && plan->desc.mask_mode == 3;
  if (needs_res && t->cmp_residual_k == nullptr) return SMLA_ERR_NULLPTR;
  if (!aligned16(t->q) || (t->k != nullptr && !aligned16(t->k))) return SMLA_ERR_INVALID;
  const void* a4[] = {wants_lse_in ? t->softmax_lse : nullptr, wants_out ? t->out : nullptr, lse_out,
                      t->sparse_indices, t->topk_length, t->seqused_q, t->seqused_k,
                      needs_res ? t->cmp_residual_k : nullptr};
  for (const void* a : a4)
    if (a != nullptr && !aligned4(a)) return SMLA_ERR_INVALID;

  // the CTA-pair kernel runs the whole-problem L1-norm launch when the plan has it
  const bool pair = mode == smla::kModeL1 && chunk < 0 && plan->pair_clusters > 0;
  CUtensorMap tq;
  const int q_box = pair ? g.G / 2 : g.R * g.G;
  if (!smla::encode_rows_map(&tq, t->q, g.q_rows, q_box, plan->desc.dtype)) {
    g_last_cuda_error = "cuTensorMapEncodeTiled(q) failed";
    return SMLA_ERR_CUDA;
  }
  smla::KernelParams p{};
  p.k = static_cast<const uint8_t*>(t->k);  // unread when there is no key row (every item has zero tiles)
  p.items = chunk < 0 ? plan->d_items : plan->d_chunk_items[chunk];
  p.cta_begin = chunk < 0 ? plan->d_cta_begin : plan->d_chunk_begin[chunk];
  p.status = plan->d_status;
  p.lse = wants_lse_in ? t->softmax_lse : nullptr;
  p.idx = g.sparse ? t->sparse_indices : nullptr;
  p.topk_len = plan->desc.has_topk_length ? t->topk_length : nullptr;
  p.seqused_q = t->seqused_q;
  p.seqused_k = t->seqused_k;
  p.out = wants_out ? t->out : nullptr;
  p.lse_out = wants_lse_in ? nullptr : lse_out;
  p.G = g.G;
  p.R = g.R;
  p.n_mma = g.n_mma;
  p.q_box_rows = q_box;
  p.topk = g.sparse ? plan->desc.topk : 0;
  p.width = g.width;
  p.mask_mode = plan->desc.mask_mode;
  p.cmp_ratio = plan->desc.cmp_ratio;
  p.cmp_res = needs_res ? t->cmp_residual_k : nullptr;
  p.stages = plan->stages;
  p.idesc = static_cast<int32_t>(plan->idesc);
  p.idesc_lse = static_cast<int32_t>(smla::make_idesc(plan->desc.dtype, smla::kTileKeys));
  p.c_log2 = static_cast<float>(static_cast<double>(plan->desc.softmax_scale) * 1.4426950408889634);
  p.inv_g = 1.0f / static_cast<float>(g.G);
  p.timeout_ns = plan->timeout_ns;
  p.withhold_q = plan->withhold_q;
  if (pair) {
    p.items = plan->d_pair_items;
    p.cta_begin = plan->d_pair_begin;
    p.stages = plan->pair_stages;
    p.idesc = static_cast<int32_t>(smla::make_idesc(plan->desc.dtype, g.n_mma, 256));
    cudaError_t e = smla::launch_pair(p, tq, plan->pair_clusters, plan->pair_smem,
                                      reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pair kernel launch");
    return SMLA_OK;
  }
  if (mode == smla::kModeL1 && chunk < 0 && plan->split_tiles > 0) {
    p.items = plan->d_split_items;
    p.cta_begin = plan->d_split_begin;
  }
  const int issuers = mode == smla::kModeL1 ? smla::l1_issuers(g) : 2;
  cudaError_t e = smla::launch_fused(p, tq, g.sparse, mode, issuers, plan->num_ctas, plan->smem,
                                     reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return SMLA_OK;
}

}  // namespace

extern "C" {

smla_status smla_l1norm_run_tensors(const smla_plan* plan, const smla_l1norm_tensors* t, smla_stream_t stream) {
  return launch_mode(plan, t, nullptr, smla::kModeL1, stream);
}

smla_status smla_softmax_lse_run(const smla_plan* plan, const smla_l1norm_tensors* t, float* lse_out,
                                 smla_stream_t stream) {
  return launch_mode(plan, t, lse_out, smla::kModeLse, stream);
}

smla_status smla_l1norm_run_fused_lse(const smla_plan* plan, const smla_l1norm_tensors* t, float* lse_out,
                                      smla_stream_t stream) {
  return launch_mode(plan, t, lse_out, smla::kModeFused, stream);
}

smla_status smla_l1norm_run(const smla_plan* plan, const void* q, const void* k, const float* softmax_lse,
                            const int32_t* sparse_indices, const int32_t* topk_length, float* out,
                            smla_stream_t stream) {
  const smla_l1norm_tensors t{q, k, softmax_lse, sparse_indices, topk_length, nullptr, nullptr, out, nullptr};
  return smla_l1norm_run_tensors(plan, &t, stream);
}

smla_status smla_l1norm_run_from_host(const smla_plan* plan, const void* h_q, const void* h_k, const float* h_lse,
                                      const int32_t* h_indices, const int32_t* h_topk_length, float* h_out,
                                      void* d_q, void* d_k, float* d_lse, int32_t* d_indices,
                                      int32_t* d_topk_length, float* d_out, smla_stream_t stream) {
  if (plan == nullptr) return SMLA_ERR_NULLPTR;
  smla_io_sizes s;
  smla_l1norm_io_sizes(plan, &s);
  auto st = reinterpret_cast<cudaStream_t>(stream);
  struct Copy {
    void* dst;
    const void* src;
    size_t n;
  } copies[5] = {{d_q, h_q, s.q_bytes},
                 {d_k, h_k, s.k_bytes},
                 {d_lse, h_lse, s.lse_bytes},
                 {d_indices, h_indices, s.indices_bytes},
                 {d_topk_length, h_topk_length, s.topk_length_bytes}};
  if (s.out_bytes > 0 && (h_out == nullptr || d_out == nullptr)) return SMLA_ERR_NULLPTR;
  for (const Copy& c : copies) {
    if (c.n == 0) continue;
    if (c.dst == nullptr || c.src == nullptr) return SMLA_ERR_NULLPTR;
  }
  const size_t n_chunks = plan->chunk_lo.size();
  if (n_chunks == 0 || plan->geo.n_tokens == 0) {
    for (const Copy& c : copies) {
      if (c.n == 0) continue;
      cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(H2D)");
    }
    smla_status r = smla_l1norm_run(plan, d_q, d_k, d_lse, d_indices, d_topk_length, d_out, stream);
    if (r != SMLA_OK) return r;
    if (s.out_bytes > 0) {
      cudaError_t e = cudaMemcpyAsync(h_out, d_out, s.out_bytes, cudaMemcpyDeviceToHost, st);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(D2H)");
    }
    return SMLA_OK;
  }
  // Pipelined over token chunks: the copy-in stream moves K, then each
  // chunk's rows of q, lse, indices and topk_length; the caller's stream
  // runs each chunk's kernel once its inputs have landed; the copy-out
  // stream returns each chunk's output rows as soon as its kernel is done.
  // H2D and D2H use different copy engines, so the only serial part is the
  // host-to-device traffic.  The caller's stream waits for the last copy.
  const smla_l1norm_tensors t{d_q, d_k, d_lse, d_indices, d_topk_length, nullptr, nullptr, d_out, nullptr};
  if (t.q == nullptr || t.softmax_lse == nullptr || t.out == nullptr) return SMLA_ERR_NULLPTR;
  const int64_t n_tok = plan->geo.n_tokens;
  auto per_token = [n_tok](size_t total) { return total / static_cast<size_t>(n_tok); };
  const Copy rows[4] = {{d_q, h_q, per_token(s.q_bytes)},
                        {d_lse, h_lse, per_token(s.lse_bytes)},
                        {d_indices, h_indices, per_token(s.indices_bytes)},
                        {d_topk_length, h_topk_length, per_token(s.topk_length_bytes)}};
  const size_t out_row = per_token(s.out_bytes);
  cudaEvent_t ev_start = plan->events[0], ev_end = plan->events[1];
  cudaError_t e = cudaEventRecord(ev_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, ev_start, 0);
  if (e == cudaSuccess && s.k_bytes > 0) e = cudaMemcpyAsync(d_k, h_k, s.k_bytes, cudaMemcpyHostToDevice, plan->s_in);
  if (e != cudaSuccess) return cuda_fail(e, "run_from_host set-up");
  for (size_t c = 0; c < n_chunks; ++c) {
    const size_t lo = static_cast<size_t>(plan->chunk_lo[c]), hi = static_cast<size_t>(plan->chunk_hi[c]);
    cudaEvent_t ev_in = plan->events[2 + 2 * c], ev_done = plan->events[3 + 2 * c];
    for (const Copy& r : rows) {
      if (r.n == 0 || hi == lo) continue;
      e = cudaMemcpyAsync(static_cast<uint8_t*>(r.dst) + lo * r.n, static_cast<const uint8_t*>(r.src) + lo * r.n,
                          (hi - lo) * r.n, cudaMemcpyHostToDevice, plan->s_in);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(H2D)");
    }
    e = cudaEventRecord(ev_in, plan->s_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
    if (e != cudaSuccess) return cuda_fail(e, "run_from_host chunk");
    const smla_status r = launch_mode(plan, &t, nullptr, smla::kModeL1, stream, static_cast<int>(c));
    if (r != SMLA_OK) return r;
    e = cudaEventRecord(ev_done, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(plan->s_out, ev_done, 0);
    if (e == cudaSuccess && out_row > 0 && hi > lo)
      e = cudaMemcpyAsync(reinterpret_cast<uint8_t*>(h_out) + lo * out_row,
                          reinterpret_cast<const uint8_t*>(d_out) + lo * out_row, (hi - lo) * out_row,
                          cudaMemcpyDeviceToHost, plan->s_out);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(D2H)");
  }
  e = cudaEventRecord(ev_end, plan->s_out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_end, 0);
  if (e != cudaSuccess) return cuda_fail(e, "run_from_host end");
  return SMLA_OK;
}

smla_status smla_l1norm_get_status(const smla_plan* plan, smla_stream_t stream, int32_t* flags) {
  if (plan == nullptr) return SMLA_ERR_NULLPTR;
  auto st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, plan->d_status, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(plan->d_status, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "get_status");
  if (flags != nullptr) *flags = v;
  if (v & smla::kFlagTimeout) return SMLA_ERR_TIMEOUT;
  if (v & smla::kFlagBadIndex) return SMLA_WARN_BAD_INDEX;
  return SMLA_OK;
}

// Test hook: run a bounded wait on a barrier that nothing completes and
// report the status it leaves (SMLA_ERR_TIMEOUT when the bound works).
smla_status smla_debug_wait_timeout_probe(int64_t timeout_ns, smla_stream_t stream, int32_t* flags) {
  int32_t* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int32_t));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(probe)");
  auto st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  e = cudaMemsetAsync(d, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = smla::launch_wait_timeout_probe(d, timeout_ns, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&v, d, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(d);
  if (e != cudaSuccess) return cuda_fail(e, "wait probe");
  if (flags != nullptr) *flags = v;
  return (v & smla::kFlagTimeout) ? SMLA_ERR_TIMEOUT : SMLA_OK;
}

smla_status smla_debug_gather(const smla_plan* plan, int32_t mode, int64_t token, const void* k,
                              const int32_t* sparse_indices, const int32_t* topk_length, void* dump,
                              int64_t dump_bytes, smla_stream_t stream) {
  if (plan == nullptr || dump == nullptr) return SMLA_ERR_NULLPTR;
  if (mode != smla::kModeL1 && mode != smla::kModeLse) return SMLA_ERR_INVALID;
  const Geometry& g = plan->geo;
  if (token < 0 || token >= g.n_tokens) return SMLA_ERR_INVALID;
  if (g.k_rows > 0 && k == nullptr) return SMLA_ERR_NULLPTR;
  if (g.sparse && sparse_indices == nullptr) return SMLA_ERR_NULLPTR;
  if (plan->desc.has_topk_length && topk_length == nullptr) return SMLA_ERR_NULLPTR;
  if ((k != nullptr && !aligned16(k)) || !aligned16(dump)) return SMLA_ERR_INVALID;
  int item = -1;
  for (size_t i = 0; i < plan->items_host.size(); ++i) {
    const WorkItem& w = plan->items_host[i];
    if (token >= w.q_tok && token < static_cast<int64_t>(w.q_tok) + w.nrows) {
      item = static_cast<int>(i);
      break;
    }
  }
  if (item < 0) return SMLA_ERR_INVALID;
  smla::KernelParams p{};
  p.k = static_cast<const uint8_t*>(k);
  p.items = plan->d_items;
  p.cta_begin = plan->d_cta_begin;
  p.status = plan->d_status;
  p.idx = g.sparse ? sparse_indices : nullptr;
  p.topk_len = plan->desc.has_topk_length ? topk_length : nullptr;
  p.G = g.G;
  p.R = g.R;
  p.n_mma = g.n_mma;
  p.q_box_rows = g.R * g.G;
  p.topk = g.sparse ? plan->desc.topk : 0;
  p.width = g.width;
  p.mask_mode = plan->desc.mask_mode;
  p.cmp_ratio = plan->desc.cmp_ratio;
  p.stages = plan->stages;
  p.timeout_ns = plan->timeout_ns;
  cudaError_t e = smla::configure_fused_for_device();
  if (e == cudaSuccess)
    e = smla::launch_gather_dump(p, g.sparse, mode, item, item + 1, static_cast<uint8_t*>(dump),
                                 dump_bytes / smla::kKStageBytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather dump");
  return SMLA_OK;
}

const char* smla_status_string(smla_status s) {
  switch (s) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_NULLPTR: return "SMLA_ERR_NULLPTR: a required pointer is NULL";
    case SMLA_ERR_INVALID: return "SMLA_ERR_INVALID: shape, layout, dtype or constraint violated";
    case SMLA_ERR_UNSUPPORTED:
      return "SMLA_ERR_UNSUPPORTED: documented feature not built (mask modes 1/2; compressed causal keys in "
             "smla_l1norm_run_noalloc)";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA: a CUDA call failed";
    case SMLA_ERR_TIMEOUT: return "SMLA_ERR_TIMEOUT: a device-side wait gave up";
    case SMLA_WARN_BAD_INDEX: return "SMLA_WARN_BAD_INDEX: a sparse index outside [-1, Sk) was treated as masked";
    case SMLA_ERR_CAPACITY:
      return "SMLA_ERR_CAPACITY: smla_l1norm_run_noalloc holds at most 65536 work items and 1024 CTAs";
  }
  return "unknown smla_status";
}

const char* smla_get_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

}  // extern "C"
