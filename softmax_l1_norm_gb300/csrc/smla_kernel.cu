// Fused Sparse-Flash-MLA Softmax-L1Norm forward for sm_103a (GB300).
//
// What it computes (article "SparseFlashMlaSoftmaxL1Norm", CANN
// ops-transformer, section 三阶段计算公式): for each query token and each
// output slot i,
//     out[i] = (1/G) * sum_g exp(scale * q[g] . K[j_i] - lse[g])   if slot i is kept
//     out[i] = 0                                                   otherwise
// with j_i = sparse_indices[i] (stage 1 gather) or j_i = i (dense form).
//
// How (one persistent CTA per SM, 384 threads, warp-specialised):
//   warp 0      producer.  TMA loads the token's q block (G heads x 512) into
//               8 shared-memory chunks of 64 columns (SWIZZLE_128B), and
//               streams the selected key rows through a ring of 16 KB stages
//               (128 keys x 64 columns): tile::gather4 TMA for sparse
//               indices (4 arbitrary rows per instruction, one instruction
//               per lane), a plain tiled TMA for the dense form.
//   warp 1      MMA issuer.  tcgen05.mma kind::f16, M = 128 keys (A = key
//               stage), N = G heads padded to 16 (B = q chunk), K = 512 in
//               32 steps of 16, fp32 accumulation in one of 4 TMEM buffers.
//   warps 4-11  two epilogue warpgroups taking alternate tiles.  Thread t
//               owns TMEM lane t, i.e. key slot t of the tile, reads its G
//               accumulator columns, and sums exp2(s*scale*log2e - lse*log2e)
//               over the heads in registers: the head reduction needs no
//               shuffles and the fp32 stores are coalesced across the warp.
// The article's kernel splits the G heads of one token across cores and
// merges them with atomic adds; here one CTA owns a token's whole G x slots
// block, so each output element is written once, in a fixed order.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the kernel
// records a timeout flag in the status word, all roles leave their loops,
// outstanding copies and MMAs are waited for (again with a limit) and the
// TMEM allocation is released.

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

// Wait for the phase with the given parity to complete, for at most
// ctl.timeout_ns, or until another role has given up.  Returns false on
// either; a timeout sets the abort flag and the status bit.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*ctl.abort) return false;
      if (global_timer_ns() - t0 > static_cast<uint64_t>(ctl.timeout_ns)) {
        *ctl.abort = 1;
        atomicOr(ctl.status, kFlagTimeout);
        return false;
      }
    }
  }
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

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Four whole rows (r0..r3) of a 2-D tensor, columns [x, x+box), into four
// consecutive 128-byte shared-memory rows; swizzle per the tensor map.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
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
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// 16 consecutive fp32 accumulator columns of this thread's TMEM lane; the
// wait is fused so the registers are only read once the load completed.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&f)[16]) {
  uint32_t v[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(v[i]);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Key tiles an item needs, and (sparse form) the clamped topk_length.
template <bool kSparse>
__device__ __forceinline__ int item_tiles(const KernelParams& p, const WorkItem& w, int& tl) {
  if (kSparse) {
    int n = p.topk;
    if (p.topk_len != nullptr) n = min(max(__ldg(p.topk_len + w.q_tok), 0), p.topk);
    if (w.Sk <= 0) n = 0;
    tl = n;
    return (n + kTileKeys - 1) / kTileKeys;
  }
  tl = 0;
  return w.ntiles;
}

}  // namespace

template <bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    smla_fused_kernel(const __grid_constant__ KernelParams p,
                      const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k) {
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
      mbar_init(bar_k_full + 8 * s, 1);
      mbar_init(bar_k_empty + 8 * s, 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bar_acc_full + 8 * b, 1);
      mbar_init(bar_acc_empty + 8 * b, 128);
    }
    mbar_init(bar_teardown, 1);
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
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kAccBufs * kAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int it0 = p.cta_begin[blockIdx.x];
  const int it1 = p.cta_begin[blockIdx.x + 1];

  if (warp == 0) {
    // ============================================================ producer
    uint32_t kst = 0, kph = 0, qit = 0;
    uint32_t k_armed = 0, k_par = 0, q_armed = 0, q_par = 0;  // for the drain on abort
    bool ok = true;
    const uint32_t q_tx = static_cast<uint32_t>(p.q_box_rows) * 128u;
    for (int it = it0; it < it1 && ok; ++it) {
      const WorkItem w = p.items[it];
      int tl;
      const int nt = item_tiles<kSparse>(p, w, tl);
      if (nt == 0) continue;
      const int64_t idx_row = static_cast<int64_t>(w.q_tok) * p.topk;
      for (int t = 0; t < nt && ok; ++t) {
        int rows[4] = {0, 0, 0, 0};
        if (kSparse) {
          bool bad = false;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int slot = t * kTileKeys + lane * 4 + i;
            int j = -1;
            if (slot < tl) j = __ldg(p.idx + idx_row + slot);
            const bool in = (j >= 0) && (j < w.Sk);
            bad |= (slot < tl) && !in && (j != -1);
            rows[i] = w.k_base + (in ? j : 0);
          }
          if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, kFlagBadIndex);
        }
        for (int c = 0; c < kNumChunks; ++c) {
          if (lane == 0) {
            if (t == 0) {
              ok = wait_bounded(bar_q_empty + 8 * c, (qit & 1u) ^ 1u, ctl);
              if (ok) {
                mbar_arrive_expect_tx(bar_q_full + 8 * c, q_tx);
                tma_load_2d(sQ + c * q_chunk_bytes, &tmap_q, c * kChunkElems, w.q_tok * p.G,
                            bar_q_full + 8 * c);
                q_armed |= 1u << c;
                q_par = (q_par & ~(1u << c)) | ((qit & 1u) << c);
              }
            }
            if (ok) ok = wait_bounded(bar_k_empty + 8 * kst, kph ^ 1u, ctl);
            if (ok) mbar_arrive_expect_tx(bar_k_full + 8 * kst, kKStageBytes);
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          const uint32_t dst = sK + kst * kKStageBytes;
          if (kSparse) {
            tma_gather4(dst + lane * 4 * 128, &tmap_k, c * kChunkElems, rows[0], rows[1], rows[2],
                        rows[3], bar_k_full + 8 * kst);
          } else if (lane == 0) {
            tma_load_2d(dst, &tmap_k, c * kChunkElems, w.k_base + t * kTileKeys,
                        bar_k_full + 8 * kst);
          }
          k_armed |= 1u << kst;
          k_par = (k_par & ~(1u << kst)) | (kph << kst);
          if (++kst == static_cast<uint32_t>(p.stages)) {
            kst = 0;
            kph ^= 1u;
          }
        }
      }
      ++qit;
    }
    if (!ok && lane == 0) {
      // Let every copy this warp started land before shared memory is released.
      for (int s = 0; s < p.stages; ++s)
        if (k_armed & (1u << s)) wait_drain(bar_k_full + 8 * s, (k_par >> s) & 1u, 100000000);
      for (int c = 0; c < kNumChunks; ++c)
        if (q_armed & (1u << c)) wait_drain(bar_q_full + 8 * c, (q_par >> c) & 1u, 100000000);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      uint32_t kst = 0, kph = 0, qit = 0, acc = 0;
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it) {
        const WorkItem w = p.items[it];
        int tl;
        const int nt = item_tiles<kSparse>(p, w, tl);
        if (nt == 0) continue;
        for (int t = 0; t < nt && ok; ++t, ++acc) {
          const uint32_t buf = acc & (kAccBufs - 1);
          const uint32_t use = acc / kAccBufs;
          ok = wait_bounded(bar_acc_empty + 8 * buf, (use & 1u) ^ 1u, ctl);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * kAccCols;
          for (int c = 0; c < kNumChunks; ++c) {
            if (t == 0) {
              ok = wait_bounded(bar_q_full + 8 * c, qit & 1u, ctl);
              if (!ok) break;
            }
            ok = wait_bounded(bar_k_full + 8 * kst, kph, ctl);
            if (!ok) break;
            tc_fence_after();
            const uint64_t a_desc = sdesc_k_major_sw128(sK + kst * kKStageBytes);
            const uint64_t b_desc = sdesc_k_major_sw128(sQ + c * q_chunk_bytes);
#pragma unroll
            for (int k = 0; k < kChunkElems / 16; ++k) {
              // advance 16 elements (32 bytes) along K inside the swizzled row
              umma_f16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, static_cast<uint32_t>(p.idesc),
                       (c | k) != 0 ? 1u : 0u);
            }
            umma_commit(bar_k_empty + 8 * kst);
            if (t == nt - 1) umma_commit(bar_q_empty + 8 * c);
            if (++kst == static_cast<uint32_t>(p.stages)) {
              kst = 0;
              kph ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(bar_acc_full + 8 * buf);
        }
        ++qit;
      }
      // All MMAs this thread issued must be complete before TMEM is released.
      umma_commit(bar_teardown);
      wait_drain(bar_teardown, 0, 200000000);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ============================================================ epilogue
    const int wg = (warp - 4) >> 2;   // warpgroup 0 or 1
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int et = quarter * 32 + lane;  // key slot inside the tile
    float* L = ltab + wg * kAccCols;
    const int bar_id = 1 + wg;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc = 0;
    int table_item = -1;
    bool ok = true;
    const float c2 = p.c_log2;
    for (int it = it0; it < it1 && ok; ++it) {
      const WorkItem w = p.items[it];
      int tl;
      const int nt = item_tiles<kSparse>(p, w, tl);
      for (int t = 0; t < nt; ++t, ++acc) {
        if (static_cast<int>(acc & 1u) != wg) continue;
        if (table_item != it) {
          // lse * log2(e) per accumulator column; +inf beyond the real heads
          // so that padded columns contribute exp2(-inf) = 0.
          wg_sync(bar_id);
          if (et < p.n_mma) {
            float v = __int_as_float(0x7f800000);
            if (et < w.nrows * p.G) v = __ldg(p.lse + static_cast<int64_t>(w.q_tok) * p.G + et) * kLog2e;
            L[et] = v;
          }
          wg_sync(bar_id);
          table_item = it;
        }
        const int slot = t * kTileKeys + et;
        bool valid = false;
        if (kSparse) {
          if (slot < tl) {
            const int j = __ldg(p.idx + static_cast<int64_t>(w.q_tok) * p.topk + slot);
            valid = (j >= 0) && (j < w.Sk) && (p.mask_mode == 0 || j <= w.r0 + w.Sk - w.Sq);
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
          float s0 = 0.f, s1 = 0.f;
          for (int c0 = 0; c0 < p.n_mma; c0 += 16) {
            float f[16];
            tmem_ld16(taddr + c0, f);
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
              s0 += fast_exp2(fmaf(f[k], c2, -L[c0 + k]));
              s1 += fast_exp2(fmaf(f[k + 1], c2, -L[c0 + k + 1]));
            }
          }
          tc_fence_before();
          mbar_arrive(bar_acc_empty + 8 * buf);
          if (slot < p.topk)
            p.out[static_cast<int64_t>(w.q_tok) * p.topk + slot] = valid ? (s0 + s1) * p.inv_g : 0.f;
        } else {
          // Dense form: columns r*G + g belong to token q_tok + r.
          const int j = slot;
          float s = 0.f;
          int g_in = 0, r = 0;
          for (int c0 = 0; c0 < p.n_mma; c0 += 16) {
            float f[16];
            tmem_ld16(taddr + c0, f);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              s += fast_exp2(fmaf(f[k], c2, -L[c0 + k]));
              if (++g_in == p.G) {
                if (r < w.nrows && j < p.width) {
                  const bool v = (j < w.Sk) &&
                                 (p.mask_mode == 0 || j <= w.r0 + r + w.Sk - w.Sq);
                  p.out[static_cast<int64_t>(w.q_tok + r) * p.width + j] = v ? s * p.inv_g : 0.f;
                }
                s = 0.f;
                g_in = 0;
                ++r;
              }
            }
          }
          tc_fence_before();
          mbar_arrive(bar_acc_empty + 8 * buf);
        }
      }
      if (!ok) break;
      // Slots past the last computed tile are zero.
      if (((it - it0) & 1) == wg) {
        if (kSparse) {
          float* o = p.out + static_cast<int64_t>(w.q_tok) * p.topk;
          for (int s = nt * kTileKeys + et; s < p.topk; s += kTileKeys) o[s] = 0.f;
        } else {
          for (int r = 0; r < w.nrows; ++r) {
            float* o = p.out + static_cast<int64_t>(w.q_tok + r) * p.width;
            for (int j = nt * kTileKeys + et; j < p.width; j += kTileKeys) o[j] = 0.f;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kAccBufs * kAccCols)
                 : "memory");
  }
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

cudaError_t configure_fused(int smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(smla_fused_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(smla_fused_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t launch_fused(const KernelParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                         bool sparse, int grid, int smem_bytes, cudaStream_t stream) {
  if (sparse)
    smla_fused_kernel<true><<<grid, kThreads, smem_bytes, stream>>>(p, tmap_q, tmap_k);
  else
    smla_fused_kernel<false><<<grid, kThreads, smem_bytes, stream>>>(p, tmap_q, tmap_k);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int32_t* status, int64_t timeout_ns, cudaStream_t stream) {
  smla_wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace smla
