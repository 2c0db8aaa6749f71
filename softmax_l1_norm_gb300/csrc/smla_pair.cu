// CTA-pair form of the sparse L1-norm launch (article "SparseFlashMlaSoftmaxL1Norm",
// section 三阶段计算公式; the same operator as smla_kernel.cu's L1-norm mode)
// for 128 heads (MMA N = 128).
//
// Two CTAs of a cluster work on the same query token.  Pair-tile p of the
// token's keys puts key tile 2p (128 keys) in the leader CTA (rank 0) and
// tile 2p + 1 in the peer (rank 1); each CTA holds its own 64 heads of q
// (the MMA's B operand is split along N between the two CTAs).  The leader's
// two MMA issuers run tcgen05.mma.cta_group::2 with M = 256: one instruction
// multiplies both CTAs' keys against all 128 heads, and each CTA's TMEM
// receives its own 128 keys x 128 heads.  Against the single-CTA kernel this
// halves the q block in shared memory (64 KB), which leaves room for a key
// ring of five 32 KB stages (two head-dim chunks each): an issuer then runs
// 8 MMAs per barrier test and commit instead of 4.
//
// Synchronisation across the pair:
//   * the leader's MMA commits go to the barriers at the same offset in both
//     CTAs (.multicast::cluster): key slot free, q chunk free, accumulator full;
//   * three relay threads in the peer forward its own "key stage full",
//     "q chunk full" and "accumulator free" phases to the leader's barriers
//     with a remote arrive, in the order the leader consumes them, so a
//     remote arrival always lands in the phase it belongs to (the peer can
//     only fill a slot again after the leader freed it);
//   * every barrier that receives an arrival from the other CTA is waited on
//     with acquire at cluster scope; every wait is bounded.
// Roles (16 warps, as the single-CTA L1-norm launch): warps 0 and 2 are the
// leader's MMA issuers and, in the peer, the key-stage and accumulator
// relays; warp 12 the peer's q relay; warp 8 the q loader; warps 4-7 the
// epilogue; the other eight warps the key producers (two groups).

#include <cstdint>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kPairHeads = 64;                          // heads of q each CTA holds
constexpr int kPairQChunkBytes = kPairHeads * 128;      // 8 KB per 64-column chunk
constexpr uint16_t kBothCtas = 0x3;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// All threads of both CTAs: earlier shared-memory writes (barrier inits)
// are visible to the other CTA afterwards.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The shared::cluster address of the same location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on a barrier of the other CTA.  Relaxed: every relay forwards a
// phase it has already observed complete (its copies landed, its TMEM loads
// waited for), after a proxy fence where the tensor cores read the data; a
// cluster-scope release here waits for the SM's memory traffic in flight and
// measured ~1,150 cycles an arrival against ~100.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// MMA across the CTA pair: A = 256 keys (128 rows in each CTA's shared
// memory at the same offset), B = the heads (half in each CTA), D in each
// CTA's TMEM at d_tmem.
template <bool kAccumulate>
__device__ __forceinline__ void umma2_f16(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                          uint32_t b_hi, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.u32 p, %6, 0;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "n"(kAccumulate ? 1 : 0)
      : "memory");
}
// Arrive on the barrier at offset `bar` in both CTAs once this thread's
// earlier pair MMAs are complete.
__device__ __forceinline__ void umma2_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(kBothCtas)
      : "memory");
}
// The same, on this CTA's barrier only.
__device__ __forceinline__ void umma2_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

struct PairBars {
  uint32_t q_full, q_empty, k_full, k_empty, acc_full, acc_empty, teardown;
};

// The leader's MMA issuer H takes the wide stages s = H and H + 2 of every
// pair-tile (head-dim chunks 2s and 2s + 1, 8 MMAs per stage, one commit),
// accumulating into its own 128-column half of the pair-tile's TMEM buffer.
// The barriers it waits on receive the peer's forwarded arrivals, so they
// are acquired at cluster scope.
template <int H>
__device__ __forceinline__ void pair_mma_issue(const KernelParams& p, uint32_t sK, uint32_t sQ, const PairBars& b,
                                               uint32_t tmem_base, int it0, int it1, const WaitCtl& ctl) {
  const uint64_t a0 = sdesc_k_major_sw128(sK);
  const uint64_t b0 = sdesc_k_major_sw128(sQ);
  const uint32_t a_hi = static_cast<uint32_t>(a0 >> 32), b_hi = static_cast<uint32_t>(b0 >> 32);
  const uint32_t k_lo0 = static_cast<uint32_t>(a0), q_lo0 = static_cast<uint32_t>(b0);
  const uint32_t b_step = static_cast<uint32_t>(kPairQChunkBytes) >> 4;
  const uint32_t S = static_cast<uint32_t>(p.stages);
  const uint32_t idesc = static_cast<uint32_t>(p.idesc);
  uint32_t kst = H, kph = 0, qit = 0, acc = 0;
  bool ok = true, ready = false, acc_ready = false;
  WorkItem w_next = it0 < it1 ? p.items[it0] : WorkItem{};
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = w_next;
    if (it + 1 < it1) w_next = p.items[it + 1];
    int tl;
    const int ntk = item_tiles<true>(p, w, tl);
    if (ntk == 0) continue;
    const int np = (ntk + 1) / 2;
    const uint32_t qpar = qit & 1u;
    for (int t = 0; t < np && ok; ++t, ++acc) {
      const uint32_t buf = acc & (kAccBufs - 1);
      if (!acc_ready) {
        ok = wait_bounded_cluster(b.acc_empty + 8 * buf, ((acc / kAccBufs) & 1u) ^ 1u, ctl);
        if (!ok) break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + buf * kAccCols + H * kHalfCols;
      const bool last = (t == np - 1);
#pragma unroll
      for (int ws = H; ws < kNumChunks / 2; ws += 2) {
        const uint32_t sl = kst, ph = kph;
        kst += 2;
        if (kst >= S) {
          kst -= S;
          kph ^= 1u;
        }
        if (!ready) {
          ok = wait_bounded_cluster(b.k_full + 8 * sl, ph, ctl);
          if (!ok) break;
        }
        if (t == 0) {
          ok = wait_bounded_cluster(b.q_full + 8 * (2 * ws), qpar, ctl) &&
               wait_bounded_cluster(b.q_full + 8 * (2 * ws + 1), qpar, ctl);
          if (!ok) break;
        }
        const bool ready_next = mbar_test_wait_cluster(b.k_full + 8 * kst, kph);
        if (ws + 2 >= kNumChunks / 2)
          acc_ready = mbar_test_wait_cluster(b.acc_empty + 8 * (buf ^ 1u), (((acc + 1) / kAccBufs) & 1u) ^ 1u);
        // this CTA's producers wrote with cp.async (generic proxy); the peer's
        // relay fenced its own CTA's stage before forwarding the arrival.
        // Fenced for every stage: skipping the fence for a stage acquired
        // before the previous fence measured no faster.
        fence_proxy_async();
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t k_lo = k_lo0 + ((sl * 2 * kKStageBytes + h * kKStageBytes) >> 4);
          const uint32_t q_lo = q_lo0 + (2 * ws + h) * b_step;
          if (ws == H && h == 0)
            umma2_f16<false>(d_tmem, k_lo, a_hi, q_lo, b_hi, idesc);
          else
            umma2_f16<true>(d_tmem, k_lo, a_hi, q_lo, b_hi, idesc);
          umma2_f16<true>(d_tmem, k_lo + 2, a_hi, q_lo + 2, b_hi, idesc);
          umma2_f16<true>(d_tmem, k_lo + 4, a_hi, q_lo + 4, b_hi, idesc);
          umma2_f16<true>(d_tmem, k_lo + 6, a_hi, q_lo + 6, b_hi, idesc);
        }
        umma2_commit_both(b.k_empty + 8 * sl);
        if (last) {
          umma2_commit_both(b.q_empty + 8 * (2 * ws));
          umma2_commit_both(b.q_empty + 8 * (2 * ws + 1));
        }
        ready = ready_next;
      }
      if (!ok) break;
      umma2_commit_both(b.acc_full + 8 * buf);
    }
    ++qit;
  }
}

// Peer relay: the peer's key stages, in the order the leader consumes them.
__device__ __forceinline__ void relay_key_stages(const KernelParams& p, const PairBars& b, int it0, int it1,
                                                 const WaitCtl& ctl) {
  const uint32_t S = static_cast<uint32_t>(p.stages);
  uint32_t slot = 0, ph = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    int tl;
    const int ntk = item_tiles<true>(p, w, tl);
    const int nstages = ((ntk + 1) / 2) * (kNumChunks / 2);  // wide stages
    for (int n = 0; n < nstages; ++n) {
      if (!wait_bounded(b.k_full + 8 * slot, ph, ctl)) return;
      // the producers' cp.async writes, acquired above, become visible to
      // the tensor cores (async proxy) that the leader's MMAs drive
      fence_proxy_async();
      mbar_arrive_remote(mapa_shared(b.k_full + 8 * slot, 0));
      if (++slot == S) {
        slot = 0;
        ph ^= 1u;
      }
    }
  }
}

// Peer relay: the peer's accumulator buffers, freed by its epilogue.
__device__ __forceinline__ void relay_accumulators(const KernelParams& p, const PairBars& b, int it0, int it1,
                                                   const WaitCtl& ctl) {
  uint32_t acc = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    int tl;
    const int np = (item_tiles<true>(p, w, tl) + 1) / 2;
    for (int t = 0; t < np; ++t, ++acc) {
      const uint32_t buf = acc & (kAccBufs - 1);
      if (!wait_bounded(b.acc_empty + 8 * buf, (acc / kAccBufs) & 1u, ctl)) return;
      mbar_arrive_remote(mapa_shared(b.acc_empty + 8 * buf, 0));
    }
  }
}

// Peer relay: the peer's q chunks of each item.
__device__ __forceinline__ void relay_q(const KernelParams& p, const PairBars& b, int it0, int it1,
                                        const WaitCtl& ctl) {
  uint32_t qit = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    int tl;
    if (item_tiles<true>(p, w, tl) == 0) continue;
    for (int c = 0; c < kNumChunks; ++c) {
      if (!wait_bounded(b.q_full + 8 * c, qit & 1u, ctl)) return;
      mbar_arrive_remote(mapa_shared(b.q_full + 8 * c, 0));
    }
    ++qit;
  }
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kernel_threads<kModeL1, 2>(), 1)
    smla_pair_kernel(const __grid_constant__ KernelParams p, const __grid_constant__ CUtensorMap tmap_q) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base;
  const uint32_t sK = sQ + kNumChunks * kPairQChunkBytes;
  const uint32_t sBar = sK + p.stages * (2 * kKStageBytes);
  PairBars bars;
  bars.q_full = sBar;
  bars.q_empty = bars.q_full + 8 * kNumChunks;
  bars.k_full = bars.q_empty + 8 * kNumChunks;
  bars.k_empty = bars.k_full + 8 * kMaxStages;
  bars.acc_full = bars.k_empty + 8 * kMaxStages;
  bars.acc_empty = bars.acc_full + 8 * kAccBufs;
  bars.teardown = bars.acc_empty + 8 * kAccBufs;
  const uint32_t sMisc = bars.teardown + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sMisc - base));
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + (sMisc - base) + 4);
  float* NL = reinterpret_cast<float*>(gbase + (sMisc - base) + 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    // the leader's barriers also count the peer's forwarded arrival
    const uint32_t fwd = leader ? 1u : 0u;
    for (int c = 0; c < kNumChunks; ++c) {
      mbar_init(bars.q_full + 8 * c, 1 + fwd);
      mbar_init(bars.q_empty + 8 * c, 1);
    }
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bars.k_full + 8 * s, producer_groups<kModeL1>() * group_warps<kModeL1>() * 32 + fwd);
      mbar_init(bars.k_empty + 8 * s, 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bars.acc_full + 8 * b, 2);  // one commit per MMA issuer
      mbar_init(bars.acc_empty + 8 * b, 128 + fwd);
    }
    mbar_init(bars.teardown, 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    // one warp of each CTA allocates the pair's accumulators together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kAccBufs * kAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  if (warp == kQWarp && lane == 0) prefetch_tmap(&tmap_q);
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int cl = static_cast<int>(cluster_id_x());
  const int it0 = p.cta_begin[cl];
  const int it1 = p.cta_begin[cl + 1];

  const int pw = producer_index<kModeL1, 2>(warp);
  if (pw >= 0) {
    // ============================================================ key producers
    produce_keys<true, kModeL1, true, true>(p, pw, lane, sK, bars.k_full, bars.k_empty, ctl, it0, it1,
                                            static_cast<int>(rank));
  } else if (warp == kQWarp) {
    // ============================================================ q loader (this CTA's 64 heads)
    if (lane == 0) {
      uint32_t qit = 0, q_armed = 0, q_par = 0;
      bool ok = true;
      int pf = it0;
      for (int it = it0; it < it1 && ok; ++it) {
        const WorkItem w = p.items[it];
        int tl;
        if (item_tiles<true>(p, w, tl) == 0) continue;
        for (; pf < it1 && pf <= it + 2; ++pf)
          for (int c = 0; c < kNumChunks; ++c)
            tma_prefetch_l2_2d(&tmap_q, c * kChunkElems, p.items[pf].q_tok * p.G + static_cast<int>(rank) * kPairHeads);
        for (int c = 0; c < kNumChunks; ++c) {
          ok = wait_bounded_cluster(bars.q_empty + 8 * c, (qit & 1u) ^ 1u, ctl);
          if (!ok) break;
          if (p.withhold_q != 0 && qit == 0 && c == 0) continue;  // test hook (see the single-CTA kernel)
          mbar_arrive_expect_tx(bars.q_full + 8 * c, kPairQChunkBytes);
          tma_load_2d(sQ + c * kPairQChunkBytes, &tmap_q, c * kChunkElems,
                      w.q_tok * p.G + static_cast<int>(rank) * kPairHeads, bars.q_full + 8 * c);
          q_armed |= 1u << c;
          q_par = (q_par & ~(1u << c)) | ((qit & 1u) << c);
        }
        ++qit;
      }
      if (!ok) {
        for (int c = 0; c < kNumChunks; ++c)
          if (q_armed & (1u << c)) wait_drain(bars.q_full + 8 * c, (q_par >> c) & 1u, 100000000);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarpA || warp == 2) {
    // ============================================================ MMA issuers (leader) / relays (peer)
    if (lane == 0) {
      if (leader) {
        if (warp == kMmaWarpA)
          pair_mma_issue<0>(p, sK, sQ, bars, tmem_base, it0, it1, ctl);
        else
          pair_mma_issue<1>(p, sK, sQ, bars, tmem_base, it0, it1, ctl);
        // every pair MMA this thread issued is complete before TMEM goes
        umma2_commit_local(bars.teardown);
        wait_drain(bars.teardown, 0, 200000000);
      } else if (warp == kMmaWarpA) {
        relay_key_stages(p, bars, it0, it1, ctl);
      } else {
        relay_accumulators(p, bars, it0, it1, ctl);
      }
    }
    __syncwarp();
  } else if (warp == 12) {
    // ============================================================ q relay (peer)
    if (lane == 0 && !leader) relay_q(p, bars, it0, it1, ctl);
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ============================================================ epilogue
    // Thread et owns TMEM lane et: key slot et of this CTA's tile of the
    // pair-tile; it sums exp2(s*scale*log2e - lse*log2e) over the 128 heads
    // (two partial accumulators, even / odd head-dim chunks).
    const int quarter = warp & 3;
    const int et = quarter * 32 + lane;
    constexpr int bar_id = 1;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc = 0;
    bool ok = true;
    const float c2 = p.c_log2;
    const uint64_t c2c2 = pack_f32x2(c2, c2);
    for (int it = it0; it < it1 && ok; ++it) {
      const WorkItem w = p.items[it];
      int tl;
      const int ntk = item_tiles<true>(p, w, tl);
      const int np = (ntk + 1) / 2;
      const EffLen e = effective_lengths(p, w);
      const int vlim = p.mask_mode == 0 ? e.Sk : causal_limit(p, w, e, w.r0);
      if (np > 0) {
        wg_sync(bar_id);
        NL[et] = -(__ldg(p.lse + static_cast<int64_t>(w.q_tok) * p.G + et) * kLog2e);
        wg_sync(bar_id);
      }
      const int32_t* idx_row = p.idx + static_cast<int64_t>(w.q_tok) * p.topk;
      for (int t = 0; t < np; ++t, ++acc) {
        const int slot = (2 * t + static_cast<int>(rank)) * kTileKeys + et;
        bool valid = false;
        if (slot < tl) {
          const int j = __ldg(idx_row + slot);
          valid = (j >= 0) && (j < vlim);
        }
        const uint32_t buf = acc & (kAccBufs - 1);
        bool got = wait_bounded_cluster(bars.acc_full + 8 * buf, (acc / kAccBufs) & 1u, ctl);
        got = wg_all(bar_id, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + buf * kAccCols;
        uint64_t s01 = 0;
        auto l1_16 = [&](const uint32_t (&fa)[16], const uint32_t (&ga)[16], int c0) {
          const float2* nl2 = reinterpret_cast<const float2*>(NL + c0);
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const float2 nl = nl2[k / 2];
            const uint64_t x = add_f32x2(pack_f32x2(__uint_as_float(fa[k]), __uint_as_float(fa[k + 1])),
                                         pack_f32x2(__uint_as_float(ga[k]), __uint_as_float(ga[k + 1])));
            float y0, y1;
            unpack_f32x2(fma_f32x2(x, c2c2, pack_f32x2(nl.x, nl.y)), y0, y1);
            s01 = add_f32x2(s01, pack_f32x2(fast_exp2(y0), fast_exp2(y1)));
          }
        };
        uint32_t fa[16], ga[16], fb[16], gb[16];
        tmem_ld16_issue(taddr, fa);
        tmem_ld16_issue(taddr + kHalfCols, ga);
        tmem_ld_wait(fa, ga);
        for (int c0 = 0; c0 < kMaxN; c0 += 32) {
          const bool has_a = c0 + 32 < kMaxN;
          tmem_ld16_issue(taddr + c0 + 16, fb);
          tmem_ld16_issue(taddr + kHalfCols + c0 + 16, gb);
          l1_16(fa, ga, c0);
          tmem_ld_wait(fb, gb);
          if (has_a) {
            tmem_ld16_issue(taddr + c0 + 32, fa);
            tmem_ld16_issue(taddr + kHalfCols + c0 + 32, ga);
          }
          l1_16(fb, gb, c0 + 16);
          if (has_a) tmem_ld_wait(fa, ga);
        }
        tc_fence_before();
        mbar_arrive(bars.acc_empty + 8 * buf);
        float s0, s1;
        unpack_f32x2(s01, s0, s1);
        if (slot < p.topk)
          p.out[static_cast<int64_t>(w.q_tok) * p.topk + slot] = valid ? (s0 + s1) * p.inv_g : 0.f;
      }
      if (!ok) break;
      // slots past the pair-tiles: this CTA zeroes every other 128-slot tile
      float* o = p.out + static_cast<int64_t>(w.q_tok) * p.topk;
      for (int s = (2 * np + static_cast<int>(rank)) * kTileKeys + et; s < p.topk; s += 2 * kTileKeys) o[s] = 0.f;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no MMA, copy or remote arrival of either CTA is still in flight
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kAccBufs * kAccCols)
                 : "memory");
  }
  cluster_sync_all();
}

int pair_smem_bytes(int stages) {
  const int q_bytes = kNumChunks * kPairQChunkBytes;
  const int ring = stages * 2 * kKStageBytes;  // wide stages of 32 KB
  const int bars = (2 * kNumChunks + 2 * kMaxStages + 2 * kAccBufs + 2) * 8;
  return 1024 + q_bytes + ring + bars + kMaxN * 4 + 64 + 128;
}

// Wide stages are filled by both producer groups in one order, so any depth
// is safe: the deepest ring that fits (5 slots of 32 KB at 227 KB).
int pair_stages(int smem_limit) {
  int st = kMaxStages / 2;
  while (st > 2 && pair_smem_bytes(st) > smem_limit) --st;
  return st;
}

cudaError_t configure_pair(int smem_optin, int* max_clusters) {
  cudaError_t e = cudaFuncSetAttribute(smla_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kernel_threads<kModeL1, 2>(), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(pair_smem_bytes(pair_stages(smem_optin)));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, smla_pair_kernel, &cfg);
}

cudaError_t launch_pair(const KernelParams& p, const CUtensorMap& tmap_q, int clusters, int smem_bytes,
                        cudaStream_t stream) {
  smla_pair_kernel<<<dim3(2 * clusters), dim3(kernel_threads<kModeL1, 2>()), smem_bytes, stream>>>(p, tmap_q);
  return cudaGetLastError();
}

}  // namespace smla
