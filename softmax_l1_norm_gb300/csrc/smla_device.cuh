// Device-side building blocks shared by the kernels of this library
// (smla_kernel.cu: the fused single-CTA kernel; smla_pair.cu: the CTA-pair
// kernel): PTX wrappers for mbarriers, copies, tcgen05 and packed fp32
// arithmetic, bounded waits, the warp roles and work-item helpers, and the
// key producers.  Internal; not part of the public ABI.
#pragma once

#include <cstdint>

#include "smla_internal.h"

namespace smla {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with acquire at cluster scope: for barriers that another CTA of
// the cluster arrives on (a remote arrive, or a multicast MMA commit).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of phase completion.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct WaitCtl {
  volatile int32_t* abort;  // CTA-wide: set once any wait gave up
  int32_t* status;          // device status word
  int64_t timeout_ns;
};

// Slow path of a bounded wait: poll until the phase completes, another role
// gave up, or the time limit passes (then set the abort flag and status bit).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                       int32_t* status, int64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > static_cast<uint64_t>(timeout_ns)) {
        *abort = 1;
        atomicOr(status, kFlagTimeout);
        return false;
      }
    }
  }
}

// Wait for the phase with the given parity to complete, for at most
// ctl.timeout_ns, or until another role has given up.  Returns false on
// either.  (mbarrier.try_wait may suspend the thread until the phase
// completes, so only a wait that is really stuck reaches the clock check.)
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, ctl.abort, ctl.status, ctl.timeout_ns);
}

// Bounded wait with acquire at cluster scope (barriers another CTA arrives on).
__device__ __noinline__ bool wait_slow_cluster(uint32_t bar, uint32_t parity, volatile int32_t* abort,
                                               int32_t* status, int64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > static_cast<uint64_t>(timeout_ns)) {
        *abort = 1;
        atomicOr(status, kFlagTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return wait_slow_cluster(bar, parity, ctl.abort, ctl.status, ctl.timeout_ns);
}

// Same, ignoring the abort flag: used after an abort to let copies and MMAs
// that are already in flight land before the CTA exits.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, int64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > static_cast<uint64_t>(limit_ns)) return false;
  }
}

// ---------------------------------------------------------------- copies
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Bring a box of a tensor into L2 ahead of its load (no shared memory used).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// 16 bytes global -> shared, cached in L2 only; with `copy` false nothing
// is read and the 16 bytes are zero-filled (src must still be a valid address).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool copy = true) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(copy ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Arrive on the barrier once every cp.async this thread has issued so far
// has landed (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Make this thread's completed generic-proxy shared-memory writes visible to
// the async proxy (the tensor cores read their operands through it).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor for a K-major operand stored as 128-byte
// rows in the 128-byte swizzle pattern, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_k_major_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                  // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride offset: 8 rows * 128 B
  d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
  return d;
}
// tcgen05.mma kind::f16 with the descriptors given as (low, high) 32-bit
// halves and a constant accumulate flag: the issuing thread's per-MMA work is
// two moves.
template <bool kAccumulate>
__device__ __forceinline__ void umma_f16_lohi(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                              uint32_t b_lo, uint32_t b_hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(kAccumulate ? 1 : 0)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// Split form for software pipelining: issue the loads of the next 16
// columns of both accumulator halves, work on the current ones, then wait.
// The wait names the in-flight registers so that no use of them moves
// above it.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]),
                 "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15])
               :
               : "memory");
  asm volatile(""
               : "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]),
                 "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]),
                 "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]));
}

// Registers written by a tcgen05.ld that an earlier tmem_ld_wait covered:
// ties them to a point after that wait so that no use moves above it.
__device__ __forceinline__ void tmem_regs_after_wait(uint32_t (&a)[16]) {
  asm volatile(""
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
                 "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]),
                 "+r"(a[14]), "+r"(a[15]));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes in one 64-bit register: Blackwell's packed f32x2
// add and fma round each lane exactly as the scalar instructions do.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Named barriers for one epilogue warpgroup (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void wg_sync(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
__device__ __forceinline__ bool wg_all(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Roles.
// Warps are spread over the four SM sub-partitions (warp % 4) so that the
// single MMA-issuing thread shares its sub-partition with as little else as
// possible: its issue rate is bound by its own instruction latency.
constexpr int kMmaWarpA = 0;        // issuer 0; sub-partition 0; also allocates TMEM
// MMA issuers.  Two issuers split each tile's head-dim chunks (even / odd),
// each accumulating into its own 128-column half of the tile's TMEM buffer.
// When the MMA N is at most 64, four issuers fit: issuer H takes the chunks
// c with c % 4 == H, each into its own 64-column quarter, one issuer on each
// sub-partition (warps 0, 2, 13, 15).
template <int kIss>
__device__ __forceinline__ int issuer_index(int warp) {
  if (warp == 0) return 0;
  if (warp == 2) return 1;
  if (kIss == 4 && warp == 13) return 2;
  if (kIss == 4 && warp == 15) return 3;
  return -1;
}
constexpr int kQWarp = 8;           // sleeps in barrier waits most of the time
// Producer groups.  A lane's cp.async.mbarrier.arrive.noinc holds the warp
// until every copy the lane issued before it has landed, so a warp keeps
// one batch of copies in flight and pays about one loaded L2 round trip per
// arrive (measured on all 152 SMs: 8 copies of 512 B per warp between
// arrives give ~7.5 B/clk per warp, 16 give ~13, whatever the ring depth).
// A group of warps fills one stage; several groups fill alternate stages
// (group g fills the head-dim chunks c with c % groups == g).  The L1-norm
// mode runs 2 groups of 4 warps in 16 warps; the LSE modes one group of 4
// in 12 warps, as their epilogue needs more registers than 16 warps leave.
// A group's next stage follows its previous one by `groups` chunks; with an
// even number of ring slots, at least `groups` of them, no full or empty
// barrier is ever two phases behind a thread that waits on it.
template <int kMode>
__host__ __device__ constexpr int producer_groups() {
  return kMode == kModeL1 ? 2 : 1;
}
template <int kMode>
__host__ __device__ constexpr int group_warps() {
  return 4;
}
template <int kMode>
__host__ __device__ constexpr int keys_per_lane() {  // 4 key rows per warp instruction
  return kTileKeys / (group_warps<kMode>() * 4);
}
static_assert(kTileKeys % 16 == 0 && kNumChunks % 4 == 0, "groups own the same chunks of every tile");
static_assert(kMinStages >= 4 && kMinStages % 2 == 0, "ring depth rule");
template <int kMode, int kIss = 2>
__host__ __device__ constexpr int kernel_threads() {
  return kMode == kModeL1 ? (kIss == 4 ? 544 : 512) : kThreads;
}
constexpr int kEpiWarp0 = 4;        // warps 4-7: one warpgroup
// Producer warp number: warps 1, 3, 9, 11 (sub-partitions 1 and 3), then,
// for a second group, 13, 15, 10, 14 (with four issuers, which take warps 13
// and 15: 10, 14, 12, 16 of a 17-warp block).
template <int kMode, int kIss = 2>
__device__ __forceinline__ int producer_index(int warp) {
  constexpr int n = producer_groups<kMode>() * group_warps<kMode>();
  int i;
  switch (warp) {
    case 1: i = 0; break;
    case 3: i = 1; break;
    case 9: i = 2; break;
    case 11: i = 3; break;
    case 13: i = kIss == 4 ? 8 : 4; break;
    case 15: i = kIss == 4 ? 8 : 5; break;
    case 10: i = kIss == 4 ? 4 : 6; break;
    case 14: i = kIss == 4 ? 5 : 7; break;
    case 12: i = kIss == 4 ? 6 : 8; break;
    case 16: i = kIss == 4 ? 7 : 8; break;
    default: i = 8;
  }
  return i < n ? i : -1;
}
static_assert(producer_groups<kModeL1>() * group_warps<kModeL1>() <= 8, "8 producer warps at most");

// Lengths of an item's sequence that take part in the computation: the
// full lengths, cut to seqused_q[b] / seqused_k[b] when those are given
// (query rows at or past Sq are all zero, keys at or past Sk are masked, and
// the right-down causal diagonal is placed on the cut lengths).
struct EffLen {
  int Sq, Sk;
};
__device__ __forceinline__ EffLen effective_lengths(const KernelParams& p, const WorkItem& w) {
  EffLen e{w.Sq, w.Sk};
  if (p.seqused_q != nullptr) e.Sq = max(0, min(e.Sq, __ldg(p.seqused_q + w.b)));
  if (p.seqused_k != nullptr) e.Sk = max(0, min(e.Sk, __ldg(p.seqused_k + w.b)));
  return e;
}

// Keys visible to local row r under mask_mode 3: key j is kept iff j <
// causal_limit.  Right-down causal ([SMLA] 约束说明): row r of Sq queries sees
// key position j <= r + Sk - Sq.  Compressed keys (cmp_ratio c > 1, [SMLA]
// 参数说明): key j stands for original positions j*c .. j*c + c - 1 of
// L = Sk*c + cmp_residual_k original positions and is kept when its whole
// block is visible, j*c + c - 1 <= r + L - Sq.
__device__ __forceinline__ int causal_limit(const KernelParams& p, const WorkItem& w, const EffLen& e, int r) {
  if (p.cmp_ratio == 1) return min(e.Sk, max(0, r + e.Sk - e.Sq + 1));
  const int c = p.cmp_ratio;
  const int res = p.cmp_res != nullptr ? min(max(__ldg(p.cmp_res + w.b), 0), c - 1) : 0;
  const int64_t d = static_cast<int64_t>(r) + static_cast<int64_t>(e.Sk) * c + res - e.Sq + 1;
  if (d <= 0) return 0;
  return static_cast<int>(min(d / c, static_cast<int64_t>(e.Sk)));
}

// Key tiles an item needs, and (sparse form) the clamped topk_length.
template <bool kSparse>
__device__ __forceinline__ int item_tiles(const KernelParams& p, const WorkItem& w, int& tl) {
  if (kSparse) {
    const EffLen e = effective_lengths(p, w);
    int n = p.topk;
    if (p.topk_len != nullptr) n = min(max(__ldg(p.topk_len + w.q_tok), 0), p.topk);
    if (e.Sk <= 0 || w.r0 >= e.Sq) n = 0;
    tl = n;
    return (n + kTileKeys - 1) / kTileKeys;
  }
  tl = 0;
  if (p.seqused_q == nullptr && p.seqused_k == nullptr) return w.ntiles;
  // keys visible to the item's last participating row, within the output
  // width, counted from the item's first key tile t0.  Cut lengths can show
  // a row more keys than the full lengths the plan sized the item for (a
  // shorter Sq moves the right-down diagonal right), so the last part of a
  // pack (or a whole pack) runs to the visible end; an earlier part of a
  // split pack stops at its own range.
  const EffLen e = effective_lengths(p, w);
  const int rows = min(w.nrows, e.Sq - w.r0);
  if (rows <= 0) return 0;
  int vis = e.Sk;
  if (p.mask_mode != 0) vis = causal_limit(p, w, e, w.r0 + rows - 1);
  vis = min(vis, p.width);
  const int n = max((vis + kTileKeys - 1) / kTileKeys - w.t0, 0);
  return w.cut_tail ? min(n, w.ntiles) : n;
}

// Passes over an item's key tiles: the LSE pass, the L1-norm pass, or both.
template <int kMode>
__host__ __device__ constexpr int passes() {
  return kMode == kModeFused ? 2 : 1;
}

// Position in a CTA's sequence of (item, key tile) pairs, skipping items
// without tiles.  t runs over every pass's tiles; ktile is the key tile.
struct TileCursor {
  int it, t, nt, ntk, tl;
  WorkItem w;
  int rank;  // CTA pair layout: this CTA's rank (it takes key tile 2t + rank)
  __device__ __forceinline__ int ktile() const { return t < ntk ? t : t - ntk; }
};

// Key tile of the cursor's step: the single-CTA layout walks an item's tiles
// (twice in the fused mode); the CTA pair layout walks pair-tiles, of which
// this CTA takes tile 2t + rank (past the item's last tile when the count is
// odd: those slots are all invalid).
template <bool kPair>
__device__ __forceinline__ int cursor_ktile(const TileCursor& c) {
  return kPair ? 2 * c.t + c.rank : c.ktile();
}

template <bool kSparse, int kMode, bool kPair = false>
__device__ __forceinline__ bool cursor_next(const KernelParams& p, TileCursor& c, int it1) {
  ++c.t;
  while (c.t >= c.nt) {
    if (++c.it >= it1) return false;
    c.w = p.items[c.it];
    c.ntk = item_tiles<kSparse>(p, c.w, c.tl);
    c.nt = kPair ? (c.ntk + 1) / 2 : c.ntk * passes<kMode>();
    c.t = 0;
  }
  return true;
}

struct MmaCtx {
  uint32_t sK, sQ;
  int q_chunk_bytes;
  uint32_t bar_q_full, bar_q_empty, bar_k_full, bar_k_empty, bar_acc_full, bar_acc_empty;
  uint32_t tmem_base;
  int it0, it1;
};

// MMA issuer H (0 or 1) handles the head-dim chunks c with c % 2 == H of
// every tile, accumulating into its own 128-column half of the tile's TMEM
// buffer; the epilogue adds the two halves.  One thread issues every MMA of
// its half.  A single thread has no other work to hide its own instruction
// latency behind, so the loop is kept minimal: the descriptors differ only
// in their low word (start address), the chunk loop is unrolled and the
// accumulate flag is a constant.
//
// The L1-norm pass puts the 128 keys of a tile on M (TMEM lanes) and the
// heads on N, so that an epilogue thread owns one key slot and sums over the
// heads.  The LSE pass swaps the operands: M = 128 q rows (heads; rows past
// R*G read neighbouring shared memory and are never used), N = the 128 keys,
// so that a thread owns one head and reduces over the keys.  Both operands
// are 128-byte-swizzled K-major tiles, so the swap only exchanges the start
// addresses and the instruction descriptor.
template <bool kSparse, int kMode, int kIss, int H>
__device__ __forceinline__ void mma_issue(const KernelParams& p, const MmaCtx& m, const WaitCtl& ctl) {
  const uint64_t a0 = sdesc_k_major_sw128(m.sK);
  const uint64_t b0 = sdesc_k_major_sw128(m.sQ);
  // both descriptors share their high word (strides, version, swizzle)
  const uint32_t a_hi = static_cast<uint32_t>(a0 >> 32), b_hi = static_cast<uint32_t>(b0 >> 32);
  const uint32_t k_lo0 = static_cast<uint32_t>(a0), q_lo0 = static_cast<uint32_t>(b0);
  const uint32_t b_step = static_cast<uint32_t>(m.q_chunk_bytes) >> 4;
  const uint32_t S = static_cast<uint32_t>(p.stages);
  // Ring slot and phase of this issuer's next stage: stage n (8 per tile,
  // tile-major) uses slot n % S, and this issuer takes every kIss-th stage.
  uint32_t kst = H, kph = 0, qit = 0, acc = 0;
  bool ok = true;
  // The barrier test for this issuer's next stage is issued before the
  // current stage's MMAs (and across tile boundaries) so that its latency
  // overlaps them; only a stage that is not ready yet costs a blocking wait.
  // The accumulator buffer of the next tile is tested the same way.  Every
  // stage gets its own proxy fence: skipping it for a stage acquired before
  // the previous fence (which already covers that stage) measured 2 % slower
  // on 128 heads.
  bool ready = false, acc_ready = false;
  WorkItem w_next = m.it0 < m.it1 ? p.items[m.it0] : WorkItem{};
  for (int it = m.it0; it < m.it1 && ok; ++it) {
    const WorkItem w = w_next;
    if (it + 1 < m.it1) w_next = p.items[it + 1];  // in flight while this item runs
    int tl;
    const int nt = item_tiles<kSparse>(p, w, tl);
    if (nt == 0) continue;
    const uint32_t qpar = qit & 1u;
    const int ntot = nt * passes<kMode>();
    for (int t = 0; t < ntot && ok; ++t, ++acc) {
      const uint32_t buf = acc & (kAccBufs - 1);
      if (!acc_ready) {
        ok = wait_bounded(m.bar_acc_empty + 8 * buf, ((acc / kAccBufs) & 1u) ^ 1u, ctl);
        if (!ok) break;
      }
      tc_fence_after();
      const uint32_t d_tmem = m.tmem_base + buf * kAccCols + H * (kAccCols / kIss);
      const bool last = (t == ntot - 1);
      const bool lse_pass = kMode != kModeL1 && t < nt;
      const uint32_t idesc = static_cast<uint32_t>(lse_pass ? p.idesc_lse : p.idesc);
#pragma unroll
      for (int c = H; c < kNumChunks; c += kIss) {
        const uint32_t sl = kst, ph = kph;
        kst += kIss;
        if (kst >= S) {
          kst -= S;
          kph ^= 1u;
        }
        if (!ready) {
          ok = wait_bounded(m.bar_k_full + 8 * sl, ph, ctl);
          if (!ok) break;
        }
        // q chunk c of a new token was freed about 8 stages ago
        if (t == 0) {
          ok = wait_bounded(m.bar_q_full + 8 * c, qpar, ctl);
          if (!ok) break;
        }
        const bool ready_next = mbar_test_wait(m.bar_k_full + 8 * kst, kph);
        if (c + kIss >= kNumChunks)
          acc_ready = mbar_test_wait(m.bar_acc_empty + 8 * (buf ^ 1u), (((acc + 1) / kAccBufs) & 1u) ^ 1u);
        // the producers' cp.async writes (generic proxy), acquired through
        // the barrier, become visible to the tensor cores (async proxy)
        fence_proxy_async();
        tc_fence_after();
        const uint32_t k_lo = k_lo0 + sl * (kKStageBytes >> 4);
        const uint32_t q_lo = q_lo0 + c * b_step;
        const uint32_t a_lo = lse_pass ? q_lo : k_lo;
        const uint32_t b_lo = lse_pass ? k_lo : q_lo;
        // 4 K-steps of 16 elements (32 bytes) inside the swizzled rows
        if (c == H)
          umma_f16_lohi<false>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc);
        else
          umma_f16_lohi<true>(d_tmem, a_lo, a_hi, b_lo, b_hi, idesc);
        umma_f16_lohi<true>(d_tmem, a_lo + 2, a_hi, b_lo + 2, b_hi, idesc);
        umma_f16_lohi<true>(d_tmem, a_lo + 4, a_hi, b_lo + 4, b_hi, idesc);
        umma_f16_lohi<true>(d_tmem, a_lo + 6, a_hi, b_lo + 6, b_hi, idesc);
        umma_commit(m.bar_k_empty + 8 * sl);
        if (last) umma_commit(m.bar_q_empty + 8 * c);
        ready = ready_next;
      }
      if (!ok) break;
      umma_commit(m.bar_acc_full + 8 * buf);
    }
    ++qit;
  }
}

// ---------------------------------------------------------------- key producers
// Producer warp pw of group grp, lane l copies 16-byte segment (l & 7)
// of key rows r0 + (l >> 3) + 4*i, i < keys_per_lane, of each of its
// group's stages (4 whole 128-byte rows per warp instruction), r0 =
// (pw % group_warps) * 128 / group_warps.  Stage n uses ring slot
// n % stages.  Each lane's copies arrive on the slot's full barrier by
// themselves when they land (cp.async.mbarrier.arrive.noinc), so a
// producer only waits for free slots.  The generic-to-async proxy fence
// the tensor cores need is executed by the MMA thread after it acquires
// the full barrier: in a producer it would also wait for the copies
// still in flight.
//
// Wide stages (kWide, the CTA-pair kernel): a ring slot holds two chunks (32
// KB); group g fills chunk 2s + g of wide stage s into the slot's half g, so
// both groups fill every stage, in order, and the slot's full barrier counts
// both groups' lanes.  Filled in one order by every group, the ring is then
// safe at any depth, odd included.
template <bool kSparse, int kMode, bool kPair = false, bool kWide = false>
__device__ __forceinline__ void produce_keys(const KernelParams& p, int pw, int lane, uint32_t sK,
                                             uint32_t bar_k_full, uint32_t bar_k_empty, const WaitCtl& ctl,
                                             int it0, int it1, int rank = 0) {
  constexpr int kGW = group_warps<kMode>();
  constexpr int kKeysPerLane = keys_per_lane<kMode>();
  const int grp = pw / kGW;
  const int seg = lane & 7;
  const int krow0 = (pw % kGW) * (kTileKeys / kGW) + (lane >> 3);
  const uint32_t S = static_cast<uint32_t>(p.stages);
  constexpr uint32_t kStep = producer_groups<kMode>();  // chunks between this group's stages
  static_assert(!kWide || producer_groups<kMode>() == 2, "wide stages take two producer groups");
  uint32_t kst = kWide ? 0u : static_cast<uint32_t>(grp), kph = 0;  // slot of this group's next stage, phase
  bool ok = true;
  TileCursor cur{it0 - 1, 0, 0, 0, 0, WorkItem{}, rank};
  bool have = cursor_next<kSparse, kMode, kPair>(p, cur, it1);
  int jn[kKeysPerLane];
  auto fetch_indices = [&](const TileCursor& c) {
#pragma unroll
    for (int i = 0; i < kKeysPerLane; ++i) {
      const int slot = cursor_ktile<kPair>(c) * kTileKeys + krow0 + 4 * i;
      if (kSparse) {
        jn[i] = slot < c.tl ? __ldg(p.idx + static_cast<int64_t>(c.w.q_tok) * p.topk + slot) : -1;
      } else {
        jn[i] = c.w.t0 * kTileKeys + slot;  // key position (the item's key range starts at tile t0)
      }
    }
  };
  if (have) fetch_indices(cur);
  const uint8_t* kseg = p.k + seg * 16;
  while (have && ok) {
    // source key rows of this tile; an invalid slot (index -1 or out of
    // range, past topk_length or topk, past the keys) is zero-filled without
    // a read (its address is kept valid: key 0 of the sequence)
    int64_t row[kKeysPerLane];
    uint32_t inmask = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kKeysPerLane; ++i) {
      const int j = jn[i];
      const bool in = (j >= 0) && (j < cur.w.Sk);
      if (kSparse) bad |= (krow0 + 4 * i + cursor_ktile<kPair>(cur) * kTileKeys < cur.tl) && !in && (j != -1);
      row[i] = static_cast<int64_t>(cur.w.k_base) + (in ? j : 0);
      inmask |= (in ? 1u : 0u) << i;
    }
    if (kSparse && __any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kFlagBadIndex);
    TileCursor nxt = cur;
    const bool have_next = cursor_next<kSparse, kMode, kPair>(p, nxt, it1);
    if (have_next) fetch_indices(nxt);  // in flight while this tile streams
    for (int c = grp; c < kNumChunks; c += kStep) {
      // in the pair layout the slot is freed by the leader CTA's MMA commit
      ok = __all_sync(0xffffffffu, kPair ? wait_bounded_cluster(bar_k_empty + 8 * kst, kph ^ 1u, ctl)
                                         : wait_bounded(bar_k_empty + 8 * kst, kph ^ 1u, ctl));
      if (!ok) break;
      const uint32_t dst = kWide ? sK + kst * (2 * kKStageBytes) + grp * kKStageBytes : sK + kst * kKStageBytes;
      const uint8_t* kc = kseg + c * (kChunkElems * 2);
#pragma unroll
      for (int i = 0; i < kKeysPerLane; ++i) {
        const int r = krow0 + 4 * i;
        cp_async_16(dst + r * 128 + ((seg ^ (r & 7)) << 4), kc + row[i] * (kHeadDim * 2), (inmask >> i) & 1u);
      }
      cp_async_arrive_noinc(bar_k_full + 8 * kst);
      kst += kWide ? 1u : kStep;
      if (kst >= S) {
        kst -= S;
        kph ^= 1u;
      }
    }
    cur = nxt;
    have = have_next;
  }
  // Copies still in flight land before shared memory is released.
  cp_async_wait_all();
}

}  // namespace

}  // namespace smla
