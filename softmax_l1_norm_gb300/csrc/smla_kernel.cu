// Fused Sparse-Flash-MLA Softmax-L1Norm forward for sm_103a (GB300).
//
// What it computes (article "SparseFlashMlaSoftmaxL1Norm", CANN
// ops-transformer, section 三阶段计算公式): for each query token and each
// output slot i,
//     out[i] = (1/G) * sum_g exp(scale * q[g] . K[j_i] - lse[g])   if slot i is kept
//     out[i] = 0                                                   otherwise
// with j_i = sparse_indices[i] (stage 1 gather) or j_i = i (dense form).
//
// How (one persistent CTA per SM, warp-specialised: 512 threads for the L1
// norm, 384 for the LSE modes):
//   key producers (warps 1, 3, 9, 11, and 13, 15, 10, 14 for the L1 norm).
//               Each 128-key tile is moved in 8 stages of 64 head-dim columns
//               (128 keys x 128 bytes = 16 KB), each stage by one group of
//               four warps (two groups take turns in the L1-norm mode).
//               Every thread copies 16-byte
//               pieces with cp.async straight into the 128-byte-swizzle
//               position the MMA descriptor expects (a warp instruction
//               covers 4 whole 128-byte key rows), so any key order costs the
//               same as a contiguous tile.  The key indices of the next tile
//               are fetched while the current tile streams.
//   warps 0, 2  MMA issuers.  tcgen05.mma kind::f16, M = 128 keys (A = key
//               stage), N = G heads padded to 16 (B = q chunk), K = 512 in
//               32 steps of 16, fp32 accumulation in TMEM.  One thread cannot
//               issue M128xN128xK16 MMAs as fast as the tensor core runs them,
//               so two threads on different sub-partitions split K: warp 0
//               takes the even 64-column chunks, warp 2 the odd ones, each into
//               its own half of the tile's 256-column TMEM buffer.
//   warp 8      q loader.  TMA loads each token's q block (G heads x 512) as
//               8 chunks of 64 columns (SWIZZLE_128B); chunk c of the next
//               token loads as soon as the last MMA of the current token has
//               read chunk c, and the next tokens' blocks are prefetched to L2.
//   warps 4-7   epilogue warpgroup.  Thread t owns TMEM lane t, i.e. key
//               slot t of the tile, adds its two partial accumulators, and sums
//               exp2(s*scale*log2e - lse*log2e) over the heads in registers:
//               the head reduction needs no shuffles and the fp32 stores are
//               coalesced across the warp.
// The article's kernel splits the G heads of one token across cores and
// merges them with atomic adds; here one CTA owns a token's whole G x slots
// block, so each output element is written once, in a fixed order.
//
// Modes (template parameter): the L1 norm from a given LSE (above); the
// forward LSE the operator consumes, computed over the same kept slots (the
// MMA issuers swap operands so that accumulator rows are q rows, and each
// epilogue thread reduces its row over the keys with a running maximum);
// and both in one launch, an LSE pass then an L1-norm pass per work item.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the kernel
// records a timeout flag in the status word, all roles leave their loops,
// outstanding copies and MMAs are waited for (again with a limit) and the
// TMEM allocation is released.

#include <cstdint>
#include <mutex>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {

template <bool kSparse, int kMode, int kIss>
__device__ __forceinline__ void fused_body(const KernelParams& p, const CUtensorMap& tmap_q) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const int q_chunk_bytes = p.n_mma * 128;
  const uint32_t sQ = base;
  const uint32_t sK = sQ + kNumChunks * q_chunk_bytes;
  const uint32_t sBar = sK + p.stages * kKStageBytes;
  const uint32_t bar_q_full = sBar;
  const uint32_t bar_q_empty = bar_q_full + 8 * kNumChunks;
  const uint32_t bar_k_full = bar_q_empty + 8 * kNumChunks;
  const uint32_t bar_k_empty = bar_k_full + 8 * kMaxStages;
  const uint32_t bar_acc_full = bar_k_empty + 8 * kMaxStages;
  const uint32_t bar_acc_empty = bar_acc_full + 8 * kAccBufs;
  const uint32_t bar_teardown = bar_acc_empty + 8 * kAccBufs;
  const uint32_t sMisc = bar_teardown + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sMisc - base));
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + (sMisc - base) + 4);
  float* ltab = reinterpret_cast<float*>(gbase + (sMisc - base) + 64);
  // slot masks of the LSE pass: 4 words (128 slots) per tile, two tiles
  volatile uint32_t* vmask = reinterpret_cast<volatile uint32_t*>(gbase + (sMisc - base) + 64 + kMaxN * 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int c = 0; c < kNumChunks; ++c) {
      mbar_init(bar_q_full + 8 * c, 1);
      mbar_init(bar_q_empty + 8 * c, 1);
    }
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar_k_full + 8 * s, group_warps<kMode>() * 32);
      mbar_init(bar_k_empty + 8 * s, 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bar_acc_full + 8 * b, kIss);   // one commit per MMA issuer
      mbar_init(bar_acc_empty + 8 * b, 128);
    }
    mbar_init(bar_teardown, kIss);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Rows of the q chunks past R*G are never written by TMA; zero them so the
  // padded MMA columns read zeros.
  if (p.q_box_rows < p.n_mma) {
    uint4* q4 = reinterpret_cast<uint4*>(gbase);
    const int n16 = kNumChunks * q_chunk_bytes / 16;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) q4[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async();
  if (warp == kMmaWarpA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kAccBufs * kAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == kQWarp && lane == 0) prefetch_tmap(&tmap_q);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int it0 = p.cta_begin[blockIdx.x];
  const int it1 = p.cta_begin[blockIdx.x + 1];

  const int pw = producer_index<kMode, kIss>(warp);
  const int iss = issuer_index<kIss>(warp);
  if (pw >= 0) {
    // ============================================================ key producers
    produce_keys<kSparse, kMode>(p, pw, lane, sK, bar_k_full, bar_k_empty, ctl, it0, it1);
  } else if (warp == kQWarp) {
    // ============================================================ q loader
    if (lane == 0) {
      uint32_t qit = 0, q_armed = 0, q_par = 0;
      bool ok = true;
      const uint32_t q_tx = static_cast<uint32_t>(p.q_box_rows) * 128u;
      int pf = it0;  // next item whose q block is prefetched into L2
      for (int it = it0; it < it1 && ok; ++it) {
        const WorkItem w = p.items[it];
        int tl;
        if (item_tiles<kSparse>(p, w, tl) == 0) continue;
        // keep the q blocks of the next two items on their way into L2
        for (; pf < it1 && pf <= it + 2; ++pf)
          for (int c = 0; c < kNumChunks; ++c)
            tma_prefetch_l2_2d(&tmap_q, c * kChunkElems, p.items[pf].q_tok * p.G);
        for (int c = 0; c < kNumChunks; ++c) {
          ok = wait_bounded(bar_q_empty + 8 * c, (qit & 1u) ^ 1u, ctl);
          if (!ok) break;
          // test hook: chunk 0 of the first item never arrives, so the MMA
          // issuers' wait for it runs out and the launch takes its abort path
          if (p.withhold_q != 0 && qit == 0 && c == 0) continue;
          mbar_arrive_expect_tx(bar_q_full + 8 * c, q_tx);
          tma_load_2d(sQ + c * q_chunk_bytes, &tmap_q, c * kChunkElems, w.q_tok * p.G, bar_q_full + 8 * c);
          q_armed |= 1u << c;
          q_par = (q_par & ~(1u << c)) | ((qit & 1u) << c);
        }
        ++qit;
      }
      if (!ok) {
        // Let every copy this thread started land before shared memory is released.
        for (int c = 0; c < kNumChunks; ++c)
          if (q_armed & (1u << c)) wait_drain(bar_q_full + 8 * c, (q_par >> c) & 1u, 100000000);
      }
    }
    __syncwarp();
  } else if (iss >= 0) {
    // ============================================================ MMA issuers
    if (lane == 0) {
      const MmaCtx m{sK, sQ, q_chunk_bytes, bar_q_full, bar_q_empty, bar_k_full, bar_k_empty,
                     bar_acc_full, bar_acc_empty, tmem_base, it0, it1};
      if (iss == 0)
        mma_issue<kSparse, kMode, kIss, 0>(p, m, ctl);
      else if (iss == 1)
        mma_issue<kSparse, kMode, kIss, 1>(p, m, ctl);
      else if (kIss == 4 && iss == 2)
        mma_issue<kSparse, kMode, kIss, (kIss == 4 ? 2 : 0)>(p, m, ctl);
      else if (kIss == 4)
        mma_issue<kSparse, kMode, kIss, (kIss == 4 ? 3 : 0)>(p, m, ctl);
      // All MMAs this thread issued must be complete before TMEM is released.
      umma_commit(bar_teardown);
      wait_drain(bar_teardown, 0, 200000000);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ============================================================ epilogue
    const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
    const int et = quarter * 32 + lane;      // TMEM lane: key slot (L1 pass) or q row (LSE pass)
    float* NL = ltab;  // -lse * log2(e) per accumulator column (L1-norm pass)
    constexpr int bar_id = 1;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc = 0;
    bool ok = true;
    const float c2 = p.c_log2;
    const uint64_t c2c2 = pack_f32x2(c2, c2);
    const float neg_inf = __int_as_float(0xff800000);
    for (int it = it0; it < it1 && ok; ++it) {
      const WorkItem w = p.items[it];
      int tl;
      const int nt = item_tiles<kSparse>(p, w, tl);
      const EffLen e = effective_lengths(p, w);
      // sparse form: the slot's key j is kept iff 0 <= j < vlim
      const int vlim = (!kSparse || p.mask_mode == 0) ? e.Sk : causal_limit(p, w, e, w.r0);
      if (kMode != kModeL1) {
        // ---------------------------------------------------- LSE pass
        // Thread et owns accumulator row et: head et % G of token
        // q_tok + et / G.  It keeps a running maximum m and sum of
        // exp2(x - m) over the kept slots, x = s * scale * log2(e), so that
        // log2 sum_i exp2(x_i) = m + log2(sum).
        int limit = 0;  // dense form: this row sees keys j < limit
        if (!kSparse) {
          const int r = et / p.G;
          if (r < min(w.nrows, e.Sq - w.r0)) {
            limit = e.Sk;
            if (p.mask_mode != 0) limit = causal_limit(p, w, e, w.r0 + r);
            limit = min(limit, p.width);
          }
        }
        float m = neg_inf, sum = 0.f;
        // sparse form: this thread's slot index, loaded one tile ahead
        const int32_t* idx_row = kSparse ? p.idx + static_cast<int64_t>(w.q_tok) * p.topk : nullptr;
        int j_next = (kSparse && nt > 0 && et < tl) ? __ldg(idx_row + et) : -1;
        for (int t = 0; t < nt; ++t, ++acc) {
          const uint32_t buf = acc & (kAccBufs - 1);
          const uint32_t mset = (acc & 1u) * 4;
          if (kSparse) {
            // the slot masks are shared: each warp publishes its 32 slots
            const int slot = t * kTileKeys + et;
            const int j = j_next;
            const bool valid = (slot < tl) && (j >= 0) && (j < vlim);
            const uint32_t bits = __ballot_sync(0xffffffffu, valid);
            if (lane == 0) vmask[mset + quarter] = bits;
            j_next = (slot + kTileKeys < tl) ? __ldg(idx_row + slot + kTileKeys) : -1;
          }
          bool got = wait_bounded(bar_acc_full + 8 * buf, (acc / kAccBufs) & 1u, ctl);
          got = wg_all(bar_id, got);  // a barrier: the slot masks are visible after it
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + lane_addr + buf * kAccCols;
          // 16 columns at a time: x = keep ? s * scale * log2(e) : -inf;
          // the running maximum moves once per 16 columns (tree maximum) and
          // the sum is split over four chains.  The loop is kept rolled: the
          // warps of all roles share the instruction cache.
          const int lim = limit - (w.t0 + t) * kTileKeys;  // dense form: columns c < lim are kept
          // Column pairs go through packed f32x2 add / mul (each lane rounded
          // as the scalar instruction rounds it).
          auto lse16 = [&](const uint32_t (&fa)[16], const uint32_t (&ga)[16], int c0, uint32_t bits16) {
            float x[16];
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              float v0, v1;
              unpack_f32x2(mul_f32x2(add_f32x2(pack_f32x2(__uint_as_float(fa[k]), __uint_as_float(fa[k + 1])),
                                               pack_f32x2(__uint_as_float(ga[k]), __uint_as_float(ga[k + 1]))),
                                     c2c2),
                           v0, v1);
              const bool keep0 = kSparse ? ((bits16 >> k) & 1u) != 0 : (c0 + k < lim);
              const bool keep1 = kSparse ? ((bits16 >> (k + 1)) & 1u) != 0 : (c0 + k + 1 < lim);
              x[k] = keep0 ? v0 : neg_inf;
              x[k + 1] = keep1 ? v1 : neg_inf;
            }
            float t8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) t8[k] = fmaxf(x[k], x[k + 8]);
            const float cm = fmaxf(fmaxf(fmaxf(t8[0], t8[4]), fmaxf(t8[1], t8[5])),
                                   fmaxf(fmaxf(t8[2], t8[6]), fmaxf(t8[3], t8[7])));
            if (cm > m) {
              sum *= fast_exp2(m - cm);  // exp2(-inf) = 0 on the first kept slot
              m = cm;
            }
            if (m != neg_inf) {
              // four chains: columns k % 4 == 0, 1 (lanes of s01) and 2, 3 (s23)
              uint64_t s01 = 0, s23 = 0;
              const uint64_t nm = pack_f32x2(-m, -m);
#pragma unroll
              for (int k = 0; k < 16; k += 4) {
                float d0, d1, d2, d3;
                unpack_f32x2(add_f32x2(pack_f32x2(x[k], x[k + 1]), nm), d0, d1);
                unpack_f32x2(add_f32x2(pack_f32x2(x[k + 2], x[k + 3]), nm), d2, d3);
                s01 = add_f32x2(s01, pack_f32x2(fast_exp2(d0), fast_exp2(d1)));
                s23 = add_f32x2(s23, pack_f32x2(fast_exp2(d2), fast_exp2(d3)));
              }
              float s0, s1, s2, s3;
              unpack_f32x2(s01, s0, s1);
              unpack_f32x2(s23, s2, s3);
              sum += (s0 + s1) + (s2 + s3);
            }
          };
          uint32_t fa[16], ga[16], fb[16], gb[16];
          tmem_ld16_issue(taddr, fa);
          tmem_ld16_issue(taddr + kHalfCols, ga);
          tmem_ld_wait(fa, ga);
#pragma unroll 1
          for (int c0 = 0; c0 < kTileKeys; c0 += 32) {
            tmem_ld16_issue(taddr + c0 + 16, fb);
            tmem_ld16_issue(taddr + kHalfCols + c0 + 16, gb);
            const uint32_t w32 = kSparse ? vmask[mset + (c0 >> 5)] : 0u;
            lse16(fa, ga, c0, w32 & 0xffffu);
            tmem_ld_wait(fb, gb);
            if (c0 + 32 < kTileKeys) {
              tmem_ld16_issue(taddr + c0 + 32, fa);
              tmem_ld16_issue(taddr + kHalfCols + c0 + 32, ga);
            }
            lse16(fb, gb, c0 + 16, w32 >> 16);
            if (c0 + 32 < kTileKeys) tmem_ld_wait(fa, ga);
          }
          tc_fence_before();
          mbar_arrive(bar_acc_empty + 8 * buf);
        }
        if (!ok) break;
        const float lse2 = sum > 0.f ? m + log2f(sum) : neg_inf;  // -inf: no kept slot
        if (et < w.nrows * p.G) p.lse_out[static_cast<int64_t>(w.q_tok) * p.G + et] = lse2 * kLn2;
        if (kMode == kModeFused && nt > 0) {
          // the L1 pass reads the LSE per accumulator column
          wg_sync(bar_id);
          if (et < p.n_mma) NL[et] = et < w.nrows * p.G ? -lse2 : neg_inf;
          wg_sync(bar_id);
        }
      }
      if (kMode == kModeLse) continue;
      // ---------------------------------------------------- L1-norm pass
      if (kMode == kModeL1 && nt > 0) {
        // -lse * log2(e) per accumulator column; -inf beyond the real heads
        // so that padded columns contribute exp2(-inf) = 0.
        wg_sync(bar_id);
        if (et < p.n_mma) {
          float v = neg_inf;
          if (et < w.nrows * p.G) v = -(__ldg(p.lse + static_cast<int64_t>(w.q_tok) * p.G + et) * kLog2e);
          NL[et] = v;
        }
        wg_sync(bar_id);
      }
      for (int t = 0; t < nt; ++t, ++acc) {
        const int slot = (w.t0 + t) * kTileKeys + et;  // t0 = 0 in the sparse form
        bool valid = false;
        if (kSparse) {
          if (slot < tl) {
            const int j = __ldg(p.idx + static_cast<int64_t>(w.q_tok) * p.topk + slot);
            valid = (j >= 0) && (j < vlim);
          }
        }
        const uint32_t buf = acc & (kAccBufs - 1);
        const uint32_t use = acc / kAccBufs;
        bool got = wait_bounded(bar_acc_full + 8 * buf, use & 1u, ctl);
        got = wg_all(bar_id, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + buf * kAccCols;
        if (kSparse) {
          // sum over the heads of exp2(s * scale * log2(e) - lse * log2(e)),
          // 16 columns at a time, the next 16 loading meanwhile; even and
          // odd columns are summed separately.  The L1-norm launch works on
          // column pairs with packed f32x2 add and fma (each lane rounded as
          // the scalar instructions round it); the fused launch keeps the
          // scalar form, which measured faster there.
          uint64_t s01 = 0;  // (0.f, 0.f)
          float s0 = 0.f, s1 = 0.f;
          auto l1_16 = [&](const uint32_t (&fa)[16], const uint32_t (&ga)[16], int c0) {
            if constexpr (kMode == kModeL1) {
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
            } else {
#pragma unroll
              for (int k = 0; k < 16; k += 2) {
                s0 += fast_exp2(fmaf(__uint_as_float(fa[k]) + __uint_as_float(ga[k]), c2, NL[c0 + k]));
                s1 += fast_exp2(fmaf(__uint_as_float(fa[k + 1]) + __uint_as_float(ga[k + 1]), c2, NL[c0 + k + 1]));
              }
            }
          };
          const int n = p.n_mma;  // a multiple of 16
          if constexpr (kIss == 4) {
            // Four partial sums of 64 columns (N <= 64), added as
            // (q0 + q1) + (q2 + q3) per 16-column group.  Two loads are in
            // flight at a time (the 17-warp block has 96 registers a
            // thread): parts 0 and 1 of the next group load while this
            // group's exponentials run.
            constexpr int kQ = kAccCols / 4;
            uint32_t qa[16], qb[16];
            uint64_t xx[8];
            tmem_ld16_issue(taddr, qa);
            tmem_ld16_issue(taddr + kQ, qb);
#pragma unroll 1
            for (int c0 = 0; c0 < n; c0 += 16) {
              tmem_ld_wait(qa, qb);
#pragma unroll
              for (int k = 0; k < 16; k += 2)
                xx[k / 2] = add_f32x2(pack_f32x2(__uint_as_float(qa[k]), __uint_as_float(qa[k + 1])),
                                      pack_f32x2(__uint_as_float(qb[k]), __uint_as_float(qb[k + 1])));
              tmem_ld16_issue(taddr + 2 * kQ + c0, qa);
              tmem_ld16_issue(taddr + 3 * kQ + c0, qb);
              tmem_ld_wait(qa, qb);
#pragma unroll
              for (int k = 0; k < 16; k += 2)
                xx[k / 2] = add_f32x2(xx[k / 2], add_f32x2(pack_f32x2(__uint_as_float(qa[k]), __uint_as_float(qa[k + 1])),
                                                           pack_f32x2(__uint_as_float(qb[k]), __uint_as_float(qb[k + 1]))));
              if (c0 + 16 < n) {
                tmem_ld16_issue(taddr + c0 + 16, qa);
                tmem_ld16_issue(taddr + kQ + c0 + 16, qb);
              }
              const float2* nl2 = reinterpret_cast<const float2*>(NL + c0);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const float2 nl = nl2[k];
                float y0, y1;
                unpack_f32x2(fma_f32x2(xx[k], c2c2, pack_f32x2(nl.x, nl.y)), y0, y1);
                s01 = add_f32x2(s01, pack_f32x2(fast_exp2(y0), fast_exp2(y1)));
              }
            }
          } else if (n == kMaxN) {
            // 128 heads: a constant trip count, unrolled, so that the loads
            // and exponentials of neighbouring chunks interleave
            uint32_t fa[16], ga[16], fb[16], gb[16];
            tmem_ld16_issue(taddr, fa);
            tmem_ld16_issue(taddr + kHalfCols, ga);
            tmem_ld_wait(fa, ga);
#pragma unroll
            for (int c0 = 0; c0 < kMaxN; c0 += 32) {
              tmem_ld16_issue(taddr + c0 + 16, fb);
              tmem_ld16_issue(taddr + kHalfCols + c0 + 16, gb);
              l1_16(fa, ga, c0);
              tmem_ld_wait(fb, gb);
              if (c0 + 32 < kMaxN) {
                tmem_ld16_issue(taddr + c0 + 32, fa);
                tmem_ld16_issue(taddr + kHalfCols + c0 + 32, ga);
              }
              l1_16(fb, gb, c0 + 16);
              if (c0 + 32 < kMaxN) tmem_ld_wait(fa, ga);
            }
          } else {
            uint32_t fa[16], ga[16], fb[16], gb[16];
            tmem_ld16_issue(taddr, fa);
            tmem_ld16_issue(taddr + kHalfCols, ga);
            tmem_ld_wait(fa, ga);
            for (int c0 = 0; c0 < n; c0 += 32) {
              const bool has_b = c0 + 16 < n;
              const bool has_a = c0 + 32 < n;
              if (has_b) {
                tmem_ld16_issue(taddr + c0 + 16, fb);
                tmem_ld16_issue(taddr + kHalfCols + c0 + 16, gb);
              }
              l1_16(fa, ga, c0);
              if (has_b) tmem_ld_wait(fb, gb);
              if (has_a) {
                tmem_ld16_issue(taddr + c0 + 32, fa);
                tmem_ld16_issue(taddr + kHalfCols + c0 + 32, ga);
              }
              if (has_b) l1_16(fb, gb, c0 + 16);
              if (has_a) tmem_ld_wait(fa, ga);
            }
          }
          tc_fence_before();
          mbar_arrive(bar_acc_empty + 8 * buf);
          if constexpr (kMode == kModeL1) unpack_f32x2(s01, s0, s1);
          if (slot < p.topk)
            p.out[static_cast<int64_t>(w.q_tok) * p.topk + slot] = valid ? (s0 + s1) * p.inv_g : 0.f;
        } else {
          // Dense form: columns r*G + g belong to token q_tok + r; 16
          // columns at a time, the next 16 loading meanwhile.  The 16
          // exponentials of a chunk are computed independently first (column
          // pairs in packed f32x2), then summed into the running token sum:
          // with G a multiple of 16 a chunk lies inside one token and is
          // summed as a tree; otherwise column by column, closing a token
          // every G columns.  Token boundaries are the same for every thread.
          const int j = slot;
          float s = 0.f;
          int g_in = 0, r = 0;
          const bool whole_chunks = (p.G & 15) == 0;
          auto store_token = [&]() {
            if (r < w.nrows && j < p.width) {
              const bool v = (w.r0 + r < e.Sq) &&
                             (j < (p.mask_mode == 0 ? e.Sk : causal_limit(p, w, e, w.r0 + r)));
              p.out[static_cast<int64_t>(w.q_tok + r) * p.width + j] = v ? s * p.inv_g : 0.f;
            }
            s = 0.f;
            g_in = 0;
            ++r;
          };
          auto dense16 = [&](const uint32_t (&fa)[16], const uint32_t (&ga)[16], int c0) {
            float e16[16];
            const float2* nl2 = reinterpret_cast<const float2*>(NL + c0);
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              const float2 nl = nl2[k / 2];
              const uint64_t x = add_f32x2(pack_f32x2(__uint_as_float(fa[k]), __uint_as_float(fa[k + 1])),
                                           pack_f32x2(__uint_as_float(ga[k]), __uint_as_float(ga[k + 1])));
              float y0, y1;
              unpack_f32x2(fma_f32x2(x, c2c2, pack_f32x2(nl.x, nl.y)), y0, y1);
              e16[k] = fast_exp2(y0);
              e16[k + 1] = fast_exp2(y1);
            }
            if (whole_chunks) {
              float t8[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) t8[k] = e16[2 * k] + e16[2 * k + 1];
              s += ((t8[0] + t8[1]) + (t8[2] + t8[3])) + ((t8[4] + t8[5]) + (t8[6] + t8[7]));
              g_in += 16;
              if (g_in == p.G) store_token();
            } else {
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                s += e16[k];
                if (++g_in == p.G) store_token();
              }
            }
          };
          const int n = p.n_mma;  // a multiple of 16
          uint32_t fa[16], ga[16], fb[16], gb[16];
          tmem_ld16_issue(taddr, fa);
          tmem_ld16_issue(taddr + kHalfCols, ga);
          tmem_ld_wait(fa, ga);
          for (int c0 = 0; c0 < n; c0 += 32) {
            const bool has_b = c0 + 16 < n;
            const bool has_a = c0 + 32 < n;
            if (has_b) {
              tmem_ld16_issue(taddr + c0 + 16, fb);
              tmem_ld16_issue(taddr + kHalfCols + c0 + 16, gb);
            }
            dense16(fa, ga, c0);
            if (has_b) tmem_ld_wait(fb, gb);
            if (has_a) {
              tmem_ld16_issue(taddr + c0 + 32, fa);
              tmem_ld16_issue(taddr + kHalfCols + c0 + 32, ga);
            }
            if (has_b) dense16(fb, gb, c0 + 16);
            if (has_a) tmem_ld_wait(fa, ga);
          }
          tc_fence_before();
          mbar_arrive(bar_acc_empty + 8 * buf);
        }
      }
      if (!ok) break;
      // Slots past the last computed tile are zero.
      if (kSparse) {
        float* o = p.out + static_cast<int64_t>(w.q_tok) * p.topk;
        for (int s = nt * kTileKeys + et; s < p.topk; s += kTileKeys) o[s] = 0.f;
      } else {
        // to the end of the row, or, for a part of a split pack that is not
        // the last, to the end of its own key range
        const int end = w.cut_tail ? min(p.width, (w.t0 + w.ntiles) * kTileKeys) : p.width;
        for (int r = 0; r < w.nrows; ++r) {
          float* o = p.out + static_cast<int64_t>(w.q_tok + r) * p.width;
          for (int j = (w.t0 + nt) * kTileKeys + et; j < end; j += kTileKeys) o[j] = 0.f;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kAccBufs * kAccCols)
                 : "memory");
  }
}

template <bool kSparse, int kMode, int kIss>
__global__ void __launch_bounds__(kernel_threads<kMode, kIss>(), 1)
    smla_fused_kernel(const __grid_constant__ KernelParams p, const __grid_constant__ CUtensorMap tmap_q) {
  fused_body<kSparse, kMode, kIss>(p, tmap_q);
}

// The L1-norm launch with four MMA issuers runs 17 warps.  Warps are dealt
// to the four sub-partitions in turn, and each sub-partition has a quarter
// of the register file: five warps on one of them leave 96 registers a
// thread.  The host still checks with the occupancy API that one block fits.
__global__ void __launch_bounds__(kernel_threads<kModeL1, 4>(), 1)
    smla_fused_kernel_l1_4iss(const __grid_constant__ KernelParams p, const __grid_constant__ CUtensorMap tmap_q) {
  fused_body<true, kModeL1, 4>(p, tmap_q);
}

// A bounded wait on a barrier that nothing completes: checks that the
// timeout path returns and reports, without hanging the GPU.
__global__ void smla_wait_timeout_probe_kernel(int32_t* status, int64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl ctl{&abort_flag, status, timeout_ns};
    wait_bounded(smem_u32(&bar), 0, ctl);
  }
  __syncthreads();
  // leave the barrier in a completed state before the CTA exits
  if (threadIdx.x == 0) mbar_arrive(smem_u32(&bar));
}

// Test hook: the key producers of one launch mode, alone, over the work
// items [it0, it1) of a schedule, running the same produce_keys code as the
// fused kernel.  Warp 0 stands in for the MMA issuers: it takes the ring
// stages in order (stage n = chunk n % 8 of key tile n / 8, in ring slot
// n % stages), copies each 16 KB stage to ``dump`` exactly as it sits in
// shared memory (128 key rows of 128 bytes, 16-byte pieces in the 128-byte
// swizzle) and frees the slot.  Stages past ``max_stages`` are consumed
// without being written.
template <bool kSparse, int kMode>
__global__ void __launch_bounds__(kernel_threads<kMode>(), 1)
    smla_gather_dump_kernel(const __grid_constant__ KernelParams p, int it0, int it1, uint8_t* dump,
                            int64_t max_stages) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sK = base;
  const uint32_t bar_k_full = sK + p.stages * kKStageBytes;
  const uint32_t bar_k_empty = bar_k_full + 8 * kMaxStages;
  volatile int32_t* abort_flag =
      reinterpret_cast<volatile int32_t*>(gbase + (bar_k_empty + 8 * kMaxStages - base));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar_k_full + 8 * s, group_warps<kMode>() * 32);
      mbar_init(bar_k_empty + 8 * s, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int pw = producer_index<kMode, 2>(warp);
  if (pw >= 0) {
    produce_keys<kSparse, kMode>(p, pw, lane, sK, bar_k_full, bar_k_empty, ctl, it0, it1);
  } else if (warp == 0) {
    const int64_t S = p.stages;
    TileCursor cur{it0 - 1, 0, 0, 0, 0, WorkItem{}};
    int64_t n = 0;
    bool ok = true;
    while (ok && cursor_next<kSparse, kMode>(p, cur, it1)) {
      for (int c = 0; c < kNumChunks; ++c, ++n) {
        const uint32_t slot = static_cast<uint32_t>(n % S);
        const uint32_t ph = static_cast<uint32_t>((n / S) & 1);
        // every lane acquires the stage, so every lane's reads see the copies
        ok = __all_sync(0xffffffffu, wait_bounded(bar_k_full + 8 * slot, ph, ctl));
        if (!ok) break;
        if (n < max_stages) {
          const uint4* src = reinterpret_cast<const uint4*>(gbase + (sK + slot * kKStageBytes - base));
          uint4* dst = reinterpret_cast<uint4*>(dump + n * kKStageBytes);
          for (int i = lane; i < kKStageBytes / 16; i += 32) dst[i] = src[i];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_k_empty + 8 * slot);
      }
    }
  }
  __syncthreads();
}

int gather_dump_smem_bytes(int stages) { return 1024 + stages * kKStageBytes + 2 * kMaxStages * 8 + 64; }

cudaError_t launch_gather_dump(const KernelParams& p, bool sparse, int mode, int it0, int it1, uint8_t* dump,
                               int64_t max_stages, cudaStream_t stream) {
  const int smem = gather_dump_smem_bytes(p.stages);
  if (mode == kModeL1) {
    const dim3 b(kernel_threads<kModeL1>());
    if (sparse)
      smla_gather_dump_kernel<true, kModeL1><<<1, b, smem, stream>>>(p, it0, it1, dump, max_stages);
    else
      smla_gather_dump_kernel<false, kModeL1><<<1, b, smem, stream>>>(p, it0, it1, dump, max_stages);
  } else if (mode == kModeLse) {
    const dim3 b(kernel_threads<kModeLse>());
    if (sparse)
      smla_gather_dump_kernel<true, kModeLse><<<1, b, smem, stream>>>(p, it0, it1, dump, max_stages);
    else
      smla_gather_dump_kernel<false, kModeLse><<<1, b, smem, stream>>>(p, it0, it1, dump, max_stages);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

namespace {
constexpr int kMaxDevices = 64;
bool four_issuers_fit[kMaxDevices] = {};
}  // namespace

cudaError_t configure_fused_for_device() {
  // Once per device, every instantiation's cap goes to the opt-in maximum;
  // a launch still asks for exactly the shared memory its plan needs.
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const void* fns[] = {
      reinterpret_cast<const void*>(smla_fused_kernel<true, kModeL1, 2>),
      reinterpret_cast<const void*>(smla_fused_kernel_l1_4iss),
      reinterpret_cast<const void*>(smla_fused_kernel<false, kModeL1, 2>),
      reinterpret_cast<const void*>(smla_fused_kernel<true, kModeLse, 2>),
      reinterpret_cast<const void*>(smla_fused_kernel<false, kModeLse, 2>),
      reinterpret_cast<const void*>(smla_fused_kernel<true, kModeFused, 2>),
      reinterpret_cast<const void*>(smla_fused_kernel<false, kModeFused, 2>),
      reinterpret_cast<const void*>(smla_gather_dump_kernel<true, kModeL1>),
      reinterpret_cast<const void*>(smla_gather_dump_kernel<false, kModeL1>),
      reinterpret_cast<const void*>(smla_gather_dump_kernel<true, kModeLse>),
      reinterpret_cast<const void*>(smla_gather_dump_kernel<false, kModeLse>)};
  for (const void* f : fns) {
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e != cudaSuccess) return e;
  }
  int blocks = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, smla_fused_kernel_l1_4iss, kernel_threads<kModeL1, 4>(),
                                                    optin);
  if (e != cudaSuccess) return e;
  four_issuers_fit[dev] = blocks >= 1;
  done[dev] = true;
  return cudaSuccess;
}

bool four_issuers_available() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  return four_issuers_fit[dev];
}

cudaError_t launch_fused(const KernelParams& p, const CUtensorMap& tmap_q, bool sparse, int mode, int issuers,
                         int grid, int smem_bytes, cudaStream_t stream) {
  const dim3 g(grid);
  const dim3 b1(kernel_threads<kModeL1, 2>()), b14(kernel_threads<kModeL1, 4>()), b(kThreads);
  if (issuers == 4) {  // the L1-norm launch, sparse form, N <= 64
    if (mode != kModeL1 || !sparse || p.n_mma > kAccCols / 4) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && four_issuers_fit[dev]) {
      smla_fused_kernel_l1_4iss<<<g, b14, smem_bytes, stream>>>(p, tmap_q);
      return cudaGetLastError();
    }
    issuers = 2;  // the 17-warp block does not fit this device: two issuers
  }
  if (issuers != 2) return cudaErrorInvalidValue;
  switch (mode * 2 + (sparse ? 1 : 0)) {
    case kModeL1 * 2 + 1: smla_fused_kernel<true, kModeL1, 2><<<g, b1, smem_bytes, stream>>>(p, tmap_q); break;
    case kModeL1 * 2: smla_fused_kernel<false, kModeL1, 2><<<g, b1, smem_bytes, stream>>>(p, tmap_q); break;
    case kModeLse * 2 + 1: smla_fused_kernel<true, kModeLse, 2><<<g, b, smem_bytes, stream>>>(p, tmap_q); break;
    case kModeLse * 2: smla_fused_kernel<false, kModeLse, 2><<<g, b, smem_bytes, stream>>>(p, tmap_q); break;
    case kModeFused * 2 + 1: smla_fused_kernel<true, kModeFused, 2><<<g, b, smem_bytes, stream>>>(p, tmap_q); break;
    case kModeFused * 2: smla_fused_kernel<false, kModeFused, 2><<<g, b, smem_bytes, stream>>>(p, tmap_q); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int32_t* status, int64_t timeout_ns, cudaStream_t stream) {
  smla_wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace smla
