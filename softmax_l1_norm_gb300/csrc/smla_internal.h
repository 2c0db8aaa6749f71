// Internal structures shared by the host API (smla_api.cpp) and the kernel
// (smla_kernel.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/smla_l1norm.h"

namespace smla {

// Head dimension fixed by the operator's constraints (D = 512).
constexpr int kHeadDim = 512;
// Keys per MMA tile (the M of one tcgen05.mma; one TMEM lane per key).
constexpr int kTileKeys = 128;
// Head-dimension slice per shared-memory stage: 64 half values = 128 bytes,
// one SWIZZLE_128B row.
constexpr int kChunkElems = 64;
constexpr int kNumChunks = kHeadDim / kChunkElems;  // 8
constexpr int kKStageBytes = kTileKeys * kChunkElems * 2;  // 16 KB
// TMEM accumulators: 2 tile buffers of 256 fp32 columns (all 512 columns);
// each buffer holds two partial sums of 128 columns (even / odd head-dim
// chunks), issued by two MMA threads.
constexpr int kAccBufs = 2;
constexpr int kAccCols = 256;
constexpr int kHalfCols = 128;
constexpr int kMaxN = 128;  // largest MMA N (R*G padded to 16)
constexpr int kMaxStages = 12;
// The key ring holds an even number of stages, at least as many as there are
// producer groups (a group's next stage is that many chunks after its
// previous one).
constexpr int kMinStages = 4;
constexpr int kThreads = 384;  // LSE modes: 2 MMA issuers, 4 key producers, one epilogue warpgroup, q loader, 1 spare

// Status word bits.
constexpr int kFlagBadIndex = 1;
constexpr int kFlagTimeout = 2;

// One unit of work: one query token (sparse form) or R consecutive tokens of
// one sequence (dense form).  32 bytes.
struct WorkItem {
  int32_t q_tok;    // first query token (global index: b*S1 + r or cu_q[b] + r)
  int32_t nrows;    // tokens in this item (1 when sparse)
  int32_t r0;       // local row of q_tok within its sequence
  int32_t k_base;   // global key row of key position 0 of the sequence
  int32_t Sq;       // query length of the sequence
  int32_t Sk;       // key length of the sequence
  int32_t ntiles;   // dense form: 128-key tiles to compute on full lengths (the rest is zero)
  int32_t b;        // batch entry (sequence) of the item
  // Dense L1-norm launch split along the keys: the item covers key tiles
  // t0 .. t0 + ntiles - 1 of its tokens.  Every output slot depends on one
  // key only, so the parts of a token pack are independent.  The last part
  // also zeroes the row past its tiles (cut_tail = 0); an earlier part
  // zeroes only what its own tiles leave uncomputed (cut_tail = 1).
  int32_t t0 = 0;
  int32_t cut_tail = 0;
  int32_t reserved0 = 0, reserved1 = 0;
};
static_assert(sizeof(WorkItem) == 48, "WorkItem is 48 bytes");

struct KernelParams {
  const uint8_t* k;           // key rows, 1024 bytes each
  const WorkItem* items;
  const int32_t* cta_begin;   // [gridDim.x + 1]
  int32_t* status;
  const float* lse;           // (tokens, G)
  const int32_t* idx;         // (tokens, topk) or null
  const int32_t* topk_len;    // (tokens) or null
  const int32_t* seqused_q;   // (batch) participating query rows per sequence, or null
  const int32_t* seqused_k;   // (batch) participating keys per sequence, or null
  const int32_t* cmp_res;     // (batch) cmp_residual_k, or null (compressed keys, mask 3)
  float* out;                 // (tokens, width); unused by the LSE-only mode
  float* lse_out;             // (tokens, G) forward LSE written by the LSE modes, else null
  int32_t G;                  // heads per key head
  int32_t R;                  // tokens per item (dense), 1 (sparse)
  int32_t n_mma;              // MMA N = pad16(R*G)
  int32_t q_box_rows;         // rows of q one TMA box moves (= R*G)
  int32_t topk;               // 0 = dense
  int32_t width;              // output row length
  int32_t mask_mode;          // 0 or 3
  int32_t cmp_ratio;          // original key positions per key of K (1 = uncompressed)
  int32_t stages;             // key ring depth
  int32_t idesc;              // tcgen05 instruction descriptor: A = keys, B = q (M 128, N n_mma)
  int32_t idesc_lse;          // the same for the LSE pass: A = q rows, B = keys (M 128, N 128)
  float c_log2;               // softmax_scale * log2(e)
  float inv_g;                // 1 / G
  int64_t timeout_ns;         // bound on every device-side wait
  int32_t withhold_q;         // test hook: never load q chunk 0 of each CTA's first item
};

// Shared-memory footprint for a given MMA N and ring depth.
inline int smem_bytes_for(int n_mma, int stages) {
  const int q_bytes = kNumChunks * n_mma * 128;
  const int ring = stages * kKStageBytes;
  const int bars = (2 * kNumChunks + 2 * kMaxStages + 2 * kAccBufs + 2) * 8;
  const int tables = kMaxN * 4 + 64;  // lse table and slot masks of the epilogue warpgroup
  return 1024 /* alignment slack */ + q_bytes + ring + bars + tables + 128;
}

// What one launch computes.
enum Mode : int {
  kModeL1 = 0,     // the L1 norm from a given LSE
  kModeLse = 1,    // the forward LSE only
  kModeFused = 2,  // the forward LSE, then the L1 norm from it, per work item
};

// Launch the fused kernel (defined in smla_kernel.cu) with 2 MMA issuers,
// or 4 (the L1-norm launch of the sparse form with N <= 64 only).
cudaError_t launch_fused(const KernelParams& p, const CUtensorMap& tmap_q, bool sparse, int mode, int issuers,
                         int grid, int smem_bytes, cudaStream_t stream);
// Raise every instantiation's dynamic shared-memory cap to the current
// device's opt-in maximum, once per device (smla_kernel.cu).  The cap only
// ever rises, so a plan built for a small footprint never lowers it under
// another plan's larger one.
cudaError_t configure_fused_for_device();
// After configure_fused_for_device(): whether the four-issuer L1-norm block
// (17 warps) fits one SM of the current device.
bool four_issuers_available();
// Test hook: the key producers of a launch mode (kModeL1 or kModeLse) alone
// over work items [it0, it1), each ring stage copied to ``dump`` as the MMA
// would read it (smla_kernel.cu).  One CTA.
cudaError_t launch_gather_dump(const KernelParams& p, bool sparse, int mode, int it0, int it1, uint8_t* dump,
                               int64_t max_stages, cudaStream_t stream);

// ---------------------------------------------------------------- host side
// Shared by the plan path (smla_api.cpp) and the allocation-free path
// (smla_noalloc.cu); none of these allocates memory of any kind.

// What a description asks for, once validated.
struct Shape {
  bool sparse = false;
  bool tnd = false;
  int G = 0;
  int R = 1;        // tokens packed per MMA (dense form), 1 (sparse)
  int n_mma = 16;   // MMA N: R*G padded to 16
  int width = 0;    // output row length
  int batch = 0;
  int64_t n_tokens = 0;
  int64_t q_rows = 0;   // rows of the 2-D (tokens*G) x 512 view of q
  int64_t k_rows = 0;
  int64_t n_items = 0;  // work items: tokens (sparse) or packs of R tokens of one sequence (dense)
};

// Every check of the article's parameter tables and constraints on a
// description; fills ``s`` on success.  No CUDA call.
smla_status check_desc(const smla_l1norm_desc* d, Shape* s);
// Keys of a sequence visible from local row r (mask_mode 3), or all of them.
// With compressed keys (cmp_ratio c > 1) the residual is read on the device;
// the host takes the largest one (c - 1), an upper bound used for sizing
// work only.
int visible_keys(int64_t r, int64_t Sq, int64_t Sk, int mask_mode, int cmp_ratio = 1);
// Deepest key ring that fits in ``smem_limit`` bytes with an even number of
// stages, at least kMinStages (the barrier phases rely on it when several
// producer groups fill the ring).
int stages_for(int n_mma, int smem_limit);
// MMA issuers of the L1-norm launch: four when the accumulator of each is at
// most 64 columns wide (sparse form, N <= 64), else two.  The ring depth rule
// is unchanged: with two producer groups filling their stages in order, an
// even depth keeps every barrier within one phase for two or four issuers.
inline int l1_issuers(const Shape& s) { return (s.sparse && s.n_mma <= kAccCols / 4) ? 4 : 2; }
// tcgen05 instruction descriptor, kind::f16, M = m (128, or 256 for a CTA
// pair), N = n_mma.
uint32_t make_idesc(int dtype, int n_mma, int m = 128);

// The CTA-pair L1-norm kernel (smla_pair.cu): sparse form with N = 128.
// Shared memory for a ring of `stages`, the deepest even ring that fits,
// the device set-up (shared-memory cap; how many 2-CTA clusters fit at once)
// and the launch (grid = 2 * clusters).
int pair_smem_bytes(int stages);
int pair_stages(int smem_limit);
cudaError_t configure_pair(int smem_optin, int* max_clusters);
cudaError_t launch_pair(const KernelParams& p, const CUtensorMap& tmap_q, int clusters, int smem_bytes,
                        cudaStream_t stream);
// 2-D (rows x 512) SWIZZLE_128B tensor map of a half-precision tensor, boxes
// of 64 columns x box_rows rows.
bool encode_rows_map(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows, int dtype);
// Bound on every device-side wait: SMLA_WAIT_TIMEOUT_MS if set (> 0), else 2 s.
int64_t wait_timeout_ns();

}  // namespace smla
