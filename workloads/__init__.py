"""Seeded synthetic inputs for the Sparse-Flash-MLA Softmax-L1Norm forward.

This module is shared by the CPU oracle (``oracle/``), the GPU tests and
``bench.py``.  It only *draws* inputs; it holds none of the operator's
arithmetic (no Q.K products, no exp, no head reduction).  Everything is
numpy with ``PCG64`` seeded generators, so the same seed gives the same bytes
on x86 and on Arm.

Shapes and dtypes follow the operator's parameter table ("SparseFlashMlaSoftmaxL1Norm",
section 参数说明):

* q            (B, S1, N1, D) "BSND" or (T1, N1, D) "TND", fp16/bf16
* k            (B, S2, N2=1, D) or (T2, N2=1, D), same dtype as q
* softmax_lse  (B, N2=1, S1, G) or (N2=1, T1, G), fp32, G = N1 / N2
* sparse_indices (B, S1, N2=1, topk) or (T1, N2=1, topk), int32, -1 = padding
* topk_length  (B, S1, N2=1) or (T1, N2=1), int32
* cu_seqlens_q / cu_seqlens_k (B+1,), int32, TND only

Half-precision tensors are kept as their raw 16-bit patterns (``uint16``);
``dtype`` says how to read them.  bf16 values are produced by rounding a
float32 draw to nearest-even; fp16 values by numpy's own float16 cast.

The softmax LSE is an *input* to the operator (the forward attention pass
produces it; its definition lives with that pass, not here).  This module
only offers ``lse_estimate``: the value the LSE takes in expectation for the
drawn distributions (q, k ~ N(0,1)), computed from |q_g|^2 and the number of
selected keys, with no Q.K product.  Tests that need the exact LSE compute
it with the oracle.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

HEAD_DIM = 512  # the only head size the operator supports (约束说明: D 仅支持 512)

__all__ = [
    "Workload", "CONFIGS", "CONFIG_NAMES", "config_names", "make_config", "make_workload",
    "bf16_bits_from_f32", "half_bits_to_f32", "visible_count", "lse_estimate",
    "default_scale",
]


# ----------------------------------------------------------------------------
# 16-bit encodings
# ----------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def f16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def half_bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode 16-bit patterns (``bf16`` or ``fp16``) to float32, exactly."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


_CHUNK = 1 << 22


def _threads() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _normal_bits(key: tuple, shape, dtype: str) -> np.ndarray:
    """N(0,1) draws rounded to ``dtype``.  The tensor is cut into fixed chunks
    of 2^22 values; chunk c is drawn from PCG64(SeedSequence(key + (c,))), so
    the bytes do not depend on how many threads fill it."""
    from concurrent.futures import ThreadPoolExecutor
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    enc = bf16_bits_from_f32 if dtype == "bf16" else f16_bits_from_f32

    def fill(c):
        s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key) + [c])))
        out[s:e] = enc(g.standard_normal(e - s, dtype=np.float32))

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def default_scale(head_dim: int = HEAD_DIM) -> float:
    """1/sqrt(D) rounded to float32 (the value every config passes)."""
    return float(np.float32(1.0 / math.sqrt(head_dim)))


# ----------------------------------------------------------------------------
# Workload container
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    layout: str                      # "BSND" or "TND"
    dtype: str                       # "bf16" or "fp16"
    G: int                           # query heads per key head (N1 / N2, N2 = 1)
    q_bits: np.ndarray               # uint16, (B,S1,G,D) or (T1,G,D)
    k_bits: np.ndarray               # uint16, (B,S2,1,D) or (T2,1,D)
    softmax_scale: float
    mask_mode: int                   # 0 none, 3 right-down causal
    sparse_indices: Optional[np.ndarray] = None   # int32 (...,1,topk)
    topk_length: Optional[np.ndarray] = None      # int32 (...,1)
    cu_seqlens_q: Optional[np.ndarray] = None     # int32 (B+1,)
    cu_seqlens_k: Optional[np.ndarray] = None
    max_seqlen_k: int = 0            # TND dense output width
    softmax_lse: Optional[np.ndarray] = None      # float32 (B,1,S1,G) / (1,T1,G)
    seed: int = 0
    note: str = ""

    # --- derived geometry -------------------------------------------------
    @property
    def head_dim(self) -> int:
        return int(self.q_bits.shape[-1])

    @property
    def topk(self) -> int:
        return 0 if self.sparse_indices is None else int(self.sparse_indices.shape[-1])

    @property
    def batch(self) -> int:
        if self.layout == "TND":
            return int(len(self.cu_seqlens_q) - 1)
        return int(self.q_bits.shape[0])

    @property
    def n_tokens(self) -> int:
        """Total query tokens (B*S1 or T1)."""
        return int(np.prod(self.q_bits.shape[:-2]))

    @property
    def max_seqlen_q(self) -> int:
        if self.layout == "TND":
            return int(np.max(np.diff(self.cu_seqlens_q))) if self.batch else 0
        return int(self.q_bits.shape[1])

    @property
    def seqlen_k_bsnd(self) -> int:
        return int(self.k_bits.shape[1]) if self.layout == "BSND" else 0

    @property
    def out_width(self) -> int:
        if self.sparse_indices is not None:
            return self.topk
        return self.max_seqlen_k if self.layout == "TND" else int(self.k_bits.shape[1])

    def out_shape(self) -> tuple:
        if self.layout == "TND":
            return (self.n_tokens, 1, self.out_width)
        return (self.batch, self.max_seqlen_q, 1, self.out_width)

    def sequences(self):
        """Yield (b, q_tok0, Sq, k_row0, Sk) per batch entry."""
        if self.layout == "TND":
            for b in range(self.batch):
                q0, q1 = int(self.cu_seqlens_q[b]), int(self.cu_seqlens_q[b + 1])
                k0, k1 = int(self.cu_seqlens_k[b]), int(self.cu_seqlens_k[b + 1])
                yield b, q0, q1 - q0, k0, k1 - k0
        else:
            S1, S2 = self.q_bits.shape[1], self.k_bits.shape[1]
            for b in range(self.batch):
                yield b, b * S1, S1, b * S2, S2

    def token_table(self) -> np.ndarray:
        """int64 (n_tokens, 5): per query token (b, r, Sq, k_row0, Sk)."""
        t = np.zeros((self.n_tokens, 5), dtype=np.int64)
        for b, q0, Sq, k0, Sk in self.sequences():
            t[q0:q0 + Sq, 0] = b
            t[q0:q0 + Sq, 1] = np.arange(Sq)
            t[q0:q0 + Sq, 2] = Sq
            t[q0:q0 + Sq, 3] = k0
            t[q0:q0 + Sq, 4] = Sk
        return t

    def lse_rows(self) -> np.ndarray:
        """softmax_lse viewed as (n_tokens, G)."""
        return self.softmax_lse.reshape(self.n_tokens, self.G)

    def valid_slot_count(self) -> int:
        """Number of (token, slot) pairs that are valid (see ``visible_count``)."""
        tab = self.token_table()
        if self.sparse_indices is None:
            vis = visible_count(tab[:, 1], tab[:, 2], tab[:, 4], self.mask_mode)
            return int(np.minimum(vis, self.out_width).sum())
        idx = self.sparse_indices.reshape(self.n_tokens, self.topk).astype(np.int64)
        Sk = tab[:, 4:5]
        ok = (idx >= 0) & (idx < Sk)
        if self.mask_mode == 3:
            ok &= idx <= (tab[:, 1:2] + Sk - tab[:, 2:3])
        if self.topk_length is not None:
            tl = self.topk_length.reshape(self.n_tokens, 1).astype(np.int64)
            ok &= np.arange(self.topk)[None, :] < tl
        return int(ok.sum())


def visible_count(r, Sq, Sk, mask_mode: int):
    """Keys a query at local row ``r`` may see: all ``Sk`` without a mask;
    with right-down causal (mask 3) keys ``j <= r + Sk - Sq``, clamped to [0, Sk]."""
    r = np.asarray(r, dtype=np.int64)
    Sk = np.asarray(Sk, dtype=np.int64)
    if mask_mode == 0:
        return np.broadcast_to(Sk, np.broadcast(r, Sk).shape).copy()
    return np.clip(r + Sk - np.asarray(Sq, dtype=np.int64) + 1, 0, Sk)


def lse_estimate(w: Workload, n_valid: np.ndarray) -> np.ndarray:
    """Expected LSE for q,k ~ N(0,1): with s = scale * q_g.k and k ~ N(0, I),
    s ~ N(0, scale^2 |q_g|^2), so E[exp(s)] = exp(scale^2 |q_g|^2 / 2) and
    LSE ~ ln(n) + scale^2 |q_g|^2 / 2.  Rows with n = 0 get -inf.
    Returns float32 (n_tokens, G)."""
    from concurrent.futures import ThreadPoolExecutor
    qb = w.q_bits.reshape(w.n_tokens, w.G, -1)
    out = np.empty((w.n_tokens, w.G), dtype=np.float32)
    s2 = float(w.softmax_scale) ** 2
    n_valid = np.asarray(n_valid, dtype=np.float64)
    step = 1024

    def part(s):
        e = min(w.n_tokens, s + step)
        qf = half_bits_to_f32(qb[s:e], w.dtype)
        qq = np.einsum("tgd,tgd->tg", qf, qf)
        with np.errstate(divide="ignore"):
            ln_n = np.log(n_valid[s:e])[:, None]
        out[s:e] = (ln_n + 0.5 * s2 * qq.astype(np.float64)).astype(np.float32)

    starts = list(range(0, w.n_tokens, step))
    with ThreadPoolExecutor(min(_threads(), max(1, len(starts)))) as ex:
        list(ex.map(part, starts))
    return out


# ----------------------------------------------------------------------------
# index generators
# ----------------------------------------------------------------------------
def _indices_uniform(rng, vis: np.ndarray, topk: int):
    """Per row: if more than ``topk`` keys are visible, ``topk`` of them drawn
    uniformly without replacement (draw order kept); else every visible key in
    a random order.  Padding is -1 and ``topk_length`` is the count."""
    n = len(vis)
    idx = np.full((n, topk), -1, dtype=np.int32)
    tl = np.minimum(vis, topk).astype(np.int32)
    for i in range(n):
        v = int(vis[i])
        if v <= 0:
            continue
        if v <= topk:
            idx[i, :v] = rng.permutation(v)
        else:
            idx[i, :] = rng.choice(v, size=topk, replace=False)
    return idx, tl


def _indices_clustered(rng, r: np.ndarray, vis: np.ndarray, topk: int,
                       n_anchor: int = 16, window: int = 512, zipf_a: float = 1.1,
                       max_rounds: int = 12):
    """Long-context clustered selection (sorted ascending per row).

    Rows that see at most ``topk`` keys take all of them.  Other rows (local
    row i, visible keys [0, i]) take the trailing window [i-window+1, i] plus
    topk-window keys from [0, i-window]: each is anchor + sign*(Zipf(a)-1),
    the anchor uniform among the seeded anchors that lie in [0, i-window]
    (uniform over that range if none do), the sign +/-1 with equal odds;
    out-of-range values and duplicates are rejected.  If ``max_rounds``
    batches of draws still leave the row short, the rest is filled uniformly
    from the unused positions."""
    n = len(vis)
    S = int(vis.max()) if n else 0
    anchors = np.sort(rng.integers(0, max(S, 1), size=n_anchor))
    idx = np.full((n, topk), -1, dtype=np.int32)
    tl = np.minimum(vis, topk).astype(np.int32)
    need = topk - window
    for t in range(n):
        v = int(vis[t])
        if v <= 0:
            continue
        if v <= topk:
            idx[t, :v] = np.arange(v, dtype=np.int32)
            continue
        i = v - 1
        hi = i - window                     # far range is [0, hi]
        elig = anchors[anchors <= hi]
        chosen = np.zeros(0, dtype=np.int64)
        for _ in range(max_rounds):
            m = 4 * need
            if len(elig):
                a = elig[rng.integers(0, len(elig), size=m)]
                off = rng.zipf(zipf_a, size=m) - 1
                sign = np.where(rng.integers(0, 2, size=m) == 1, 1, -1)
                with np.errstate(over="ignore"):
                    cand = a + sign * np.minimum(off, np.int64(1) << 40)
            else:
                cand = rng.integers(0, hi + 1, size=m)
            cand = cand[(cand >= 0) & (cand <= hi)]
            allc = np.concatenate([chosen, cand])
            _, first = np.unique(allc, return_index=True)
            chosen = allc[np.sort(first)][:need]
            if len(chosen) >= need:
                break
        if len(chosen) < need:
            used = np.zeros(hi + 1, dtype=bool)
            used[chosen] = True
            rest = np.flatnonzero(~used)
            fill = rng.choice(rest, size=need - len(chosen), replace=False)
            chosen = np.concatenate([chosen, fill])
        row = np.concatenate([chosen, np.arange(i - window + 1, i + 1)])
        idx[t, :] = np.sort(row).astype(np.int32)
    return idx, tl


# ----------------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------------
def make_workload(*, name="custom", layout="BSND", dtype="bf16", B=1, S1=16, S2=256,
                  seqlens_q=None, seqlens_k=None, G=8, D=HEAD_DIM, topk=32,
                  mask_mode=0, index_mode="uniform", with_topk_length=True,
                  max_seqlen_k=None, seed=0, scale=None, lse="estimate",
                  rng=None, note="") -> Workload:
    """Build a seeded workload.

    ``topk=0`` means the dense (no sparse_indices) form.  ``index_mode`` is
    ``"uniform"`` (uniform among visible keys) or ``"clustered"`` (the
    long-context window + anchor scheme).  ``lse`` is ``"estimate"`` (see
    ``lse_estimate``) or ``None`` (left unset, for the caller to fill, e.g.
    with the oracle's exact LSE).  For TND pass ``seqlens_q``/``seqlens_k``.
    """
    rng = rng or np.random.Generator(np.random.PCG64(seed))
    if layout == "TND":
        seqlens_q = np.asarray(seqlens_q, dtype=np.int64)
        seqlens_k = np.asarray(seqlens_k if seqlens_k is not None else seqlens_q, dtype=np.int64)
        cu_q = np.concatenate([[0], np.cumsum(seqlens_q)]).astype(np.int32)
        cu_k = np.concatenate([[0], np.cumsum(seqlens_k)]).astype(np.int32)
        T1, T2 = int(cu_q[-1]), int(cu_k[-1])
        q_shape, k_shape = (T1, G, D), (T2, 1, D)
        if max_seqlen_k is None:
            max_seqlen_k = int(seqlens_k.max()) if len(seqlens_k) else 0
    else:
        cu_q = cu_k = None
        q_shape, k_shape = (B, S1, G, D), (B, S2, 1, D)
        max_seqlen_k = 0 if max_seqlen_k is None else max_seqlen_k
    q_bits = _normal_bits((seed, 1), q_shape, dtype)
    k_bits = _normal_bits((seed, 2), k_shape, dtype)
    w = Workload(name=name, layout=layout, dtype=dtype, G=G, q_bits=q_bits, k_bits=k_bits,
                 softmax_scale=default_scale(D) if scale is None else float(np.float32(scale)),
                 mask_mode=mask_mode, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                 max_seqlen_k=int(max_seqlen_k), seed=seed, note=note)
    tab = w.token_table()
    vis = visible_count(tab[:, 1], tab[:, 2], tab[:, 4], mask_mode)
    if topk > 0:
        if index_mode == "uniform":
            idx, tl = _indices_uniform(rng, vis, topk)
        elif index_mode == "clustered":
            idx, tl = _indices_clustered(rng, tab[:, 1], vis, topk)
        else:
            raise ValueError(index_mode)
        lead = q_shape[:-2]
        w.sparse_indices = idx.reshape(*lead, 1, topk)
        w.topk_length = tl.reshape(*lead, 1) if with_topk_length else None
        n_valid = tl
    else:
        n_valid = np.minimum(vis, w.out_width)
    if lse == "estimate":
        est = lse_estimate(w, n_valid)
        w.softmax_lse = _lse_to_layout(w, est)
    return w


def _lse_to_layout(w: Workload, rows: np.ndarray) -> np.ndarray:
    """(n_tokens, G) -> (B,1,S1,G) or (1,T1,G)."""
    rows = np.ascontiguousarray(rows, dtype=np.float32)
    if w.layout == "TND":
        return rows.reshape(1, w.n_tokens, w.G)
    return rows.reshape(w.batch, 1, w.max_seqlen_q, w.G)


def set_lse_rows(w: Workload, rows: np.ndarray) -> None:
    """Replace the whole softmax_lse from an (n_tokens, G) array."""
    w.softmax_lse = _lse_to_layout(w, rows)


# ----------------------------------------------------------------------------
# the five named configurations
# ----------------------------------------------------------------------------
CONFIG_NAMES = {
    1: "tiny_sparse_B1_S16_S2_256_G8_topk32",
    2: "dense_causal_B2_S512_G16",
    3: "dsv32_sparse_causal_S4096_G128_topk2048",
    4: "varlen_tnd_8seq_G64_topk2048",
    5: "long_clustered_S32768_G128_topk2048",
}


def _cfg_tiny_sparse(lse="estimate"):
    return make_workload(name=CONFIG_NAMES[1], layout="BSND", dtype="bf16",
                         B=1, S1=16, S2=256, G=8, topk=32, mask_mode=0, seed=1, lse=lse)


def _cfg_dense_causal(lse="estimate"):
    return make_workload(name=CONFIG_NAMES[2], layout="BSND", dtype="fp16",
                         B=2, S1=512, S2=512, G=16, topk=0, mask_mode=3, seed=2, lse=lse)


def _cfg_dsv32(lse="estimate"):
    return make_workload(name=CONFIG_NAMES[3], layout="BSND",
                         dtype="bf16", B=1, S1=4096, S2=4096, G=128, topk=2048, mask_mode=3,
                         seed=3, lse=lse)


def _cfg_varlen_tnd(lse="estimate"):
    rng = np.random.Generator(np.random.PCG64(4))
    lens = rng.integers(512, 8192, size=8, endpoint=True)
    return make_workload(name=CONFIG_NAMES[4], layout="TND", dtype="fp16",
                         seqlens_q=lens, seqlens_k=lens, G=64, topk=2048, mask_mode=3,
                         seed=4, rng=rng, lse=lse)


def _cfg_long_clustered(lse="estimate"):
    return make_workload(name=CONFIG_NAMES[5], layout="BSND", dtype="bf16",
                         B=1, S1=32768, S2=32768, G=128, topk=2048, mask_mode=3,
                         index_mode="clustered", seed=5, lse=lse)


CONFIGS = {
    1: _cfg_tiny_sparse,
    2: _cfg_dense_causal,
    3: _cfg_dsv32,
    4: _cfg_varlen_tnd,
    5: _cfg_long_clustered,
}


def config_names():
    return dict(CONFIG_NAMES)


def make_config(n: int, lse="estimate", seq_len=None) -> Workload:
    """Workload for configuration ``n`` (1..5).  ``seq_len`` shortens the
    square BSND configurations 3 and 5 (S1 = S2 = seq_len, same recipe and
    seed; named with the length) -- a smaller case of the same workload, for
    profiling captures that must stay small."""
    if seq_len is None:
        return CONFIGS[n](lse=lse)
    if n not in (3, 5):
        raise ValueError("seq_len applies to configurations 3 and 5")
    S = int(seq_len)
    if n == 3:
        return make_workload(name=f"dsv32_sparse_causal_S{S}_G128_topk2048", layout="BSND", dtype="bf16",
                             B=1, S1=S, S2=S, G=128, topk=2048, mask_mode=3, seed=3, lse=lse)
    return make_workload(name=f"long_clustered_S{S}_G128_topk2048", layout="BSND", dtype="bf16",
                         B=1, S1=S, S2=S, G=128, topk=2048, mask_mode=3, index_mode="clustered", seed=5,
                         lse=lse)
