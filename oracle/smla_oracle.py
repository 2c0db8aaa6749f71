"""Plain fp64 CPU oracle of the Sparse-Flash-MLA Softmax-L1Norm forward.

TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct statement
of what the operator computes; the GPU library is checked against it.  It
shares no code with the GPU path (no common helpers, tables or headers) and
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import it.

Source of the definition: the article "SparseFlashMlaSoftmaxL1Norm" on the
CANN ops-transformer operator library (cited below as [SMLA]).  Its section
三阶段计算公式 (three-stage formula) defines the operator:

  stage 1  selectedKv = Gather(K, sparseIndices[i]) for the selected blocks,
           or the whole K when there are no sparse indices;
  stage 2  P = SimpleSoftmax(Mask(Q . selectedKv^T . scale), softmaxLse);
  stage 3  softmaxL1Norm = ReduceSum(P, dimG) / G,  G = N1 / N2;

and its description of the vector function ``_muls_sel_vf_pse_type1_inner``
fixes the order inside stage 2: multiply by scale, then ``exp_sub`` against
the LSE, then sum over the head group and multiply by 1/G.

Readings taken where the article is silent or garbled (each is listed with
its reason in the design notes of this repository):

  R1  stage-1 bound: slot i runs over 0 <= i < topk, topk being the last
      dimension of sparse_indices (the formula's "0 <= i selectBlockCount"
      lost its "<"); with cmp_ratio = 1 a block is one key row.
  R2  SimpleSoftmax(x, lse) = exp(x - lse) with x the scaled, masked logit
      and natural logarithms (the kernel walk-through: muls, then exp_sub).
  R3  output last dimension: topk slots in slot order when sparse_indices is
      given (infershape takes K from sparse_indices' last dim), else the key
      length (BSND: S2; TND: max_seqlen_k).
  R4  TND output is (T1, N2, width); in dense TND, column j is key position j
      of the row's own sequence and columns j >= that sequence's length are 0.
  R5  an invalid slot gives exactly 0: index -1 or outside [0, Sk), slot
      i >= topk_length (when topk_length is given), or a key hidden by the
      mask.  Masked logits are -inf, and exp(-inf - lse) is 0 for any finite
      lse; the oracle writes the 0 directly so that a row with no valid slot
      (lse = -inf) is 0 rather than exp(-inf + inf).
  R6  mask_mode 3 ("rightDownCausal", the lower triangle divided at the
      right-bottom vertex): query row r of a sequence with Sq queries and Sk
      keys sees key position j iff j <= r + Sk - Sq.  In sparse mode the mask
      tests the key position j = sparse_indices[r, i], not the slot i.
  R7  TND sparse indices are positions inside the row's own sequence: key
      row = cu_seqlens_k[b] + j.
  R8  GQA head mapping n1 = n2 * G + g; with N2 = 1, g = n1.
  R9  stage 3 divides by G in fp64 (the GPU multiplies by fp32 1/G; the two
      agree within the stated tolerance and exactly for power-of-two G).
  R10 the result is rounded once, to nearest float32.
  R11 seqused_q / seqused_k (parameter table: the number of q / k tokens of
      each batch entry that actually take part in the computation): the
      sequence's effective lengths become Sq' = min(Sq, seqused_q[b]) and
      Sk' = min(Sk, seqused_k[b]); query rows r >= Sq' are all 0, keys
      j >= Sk' are masked, and mask_mode 3 uses the effective lengths
      (j <= r + Sk' - Sq').
  R12 compressed keys (parameter table: cmp_ratio, the compression rate of k,
      1..128; cmp_residual_k, per batch entry the remainder of S2 // cmpRatio,
      required when mask_mode = 3 and cmp_ratio != 1; the TND example passes
      a K of T2 rows with cmp_ratio 128 and expects an output T2 wide, so K
      holds the compressed keys).  With ratio c, key j of a sequence stands for
      the original key positions j*c .. j*c + c - 1 of an original sequence of
      L = Sk*c + res positions, res = cmp_residual_k[b] (clamped to 0..c-1;
      0 when not given).  mask_mode 3 applies the right-down causal rule to
      original positions and keeps key j only when its whole block is
      visible: j*c + c - 1 <= r + L - Sq (the article leaves the rule for a
      partly visible block open; this reading never lets a query see a block
      that holds a later position).  With c = 1 this is reading R6; with
      mask_mode 0 the ratio does not matter.  Under seqused_k, Sk is the cut
      key count and L = Sk'*c + res.

Inputs are the rounded half-precision tensors as raw 16-bit patterns plus a
dtype tag; every product and sum is carried out in float64.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

__all__ = [
    "decode_half", "token_geometry", "slot_key_positions", "slot_valid",
    "simple_softmax", "reduce_sum_g_mean", "softmax_l1_norm",
    "softmax_l1_norm_rows", "softmax_lse", "original_key_length",
]


# ----------------------------------------------------------------------------
# input decoding
# ----------------------------------------------------------------------------
def decode_half(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float64.  bf16 is the top half of an IEEE float32;
    fp16 is IEEE binary16 ([SMLA] 参数说明: q, k are FLOAT16 or BFLOAT16)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    raise ValueError(f"dtype must be 'bf16' or 'fp16', got {dtype!r}")


# ----------------------------------------------------------------------------
# geometry: which sequence a query token belongs to ([SMLA] 参数说明, shape notes)
# ----------------------------------------------------------------------------
def token_geometry(layout: str, q_shape, k_shape, cu_seqlens_q=None, cu_seqlens_k=None):
    """Return a list with one tuple (b, r, Sq, k_row0, Sk) per query token.

    BSND: q (B,S1,N1,D), k (B,S2,1,D); token t = b*S1 + r, key rows b*S2 + j.
    TND:  q (T1,N1,D), k (T2,1,D); sequence b spans tokens
          cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key rows
          cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 (the cumulative-sum form of
          the per-batch lengths).
    """
    out = []
    if layout == "BSND":
        B, S1 = int(q_shape[0]), int(q_shape[1])
        S2 = int(k_shape[1])
        for b in range(B):
            for r in range(S1):
                out.append((b, r, S1, b * S2, S2))
    elif layout == "TND":
        cq = [int(x) for x in cu_seqlens_q]
        ck = [int(x) for x in cu_seqlens_k]
        for b in range(len(cq) - 1):
            Sq, Sk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
            for r in range(Sq):
                out.append((b, r, Sq, ck[b], Sk))
    else:
        raise ValueError(f"layout must be BSND or TND, got {layout!r}")
    return out


# ----------------------------------------------------------------------------
# stage 1: which key each output slot refers to ([SMLA] 三阶段计算公式, stage 1)
# ----------------------------------------------------------------------------
def slot_key_positions(idx_row: Optional[np.ndarray], width: int) -> np.ndarray:
    """Key position j for each output slot.  Sparse: j = sparse_indices[row, i]
    for 0 <= i < topk (reading R1).  Dense: selectedKv = K, so slot j is key j."""
    if idx_row is None:
        return np.arange(width, dtype=np.int64)
    return np.asarray(idx_row, dtype=np.int64).reshape(-1)


def slot_valid(j: np.ndarray, *, r: int, Sq: int, Sk: int, mask_mode: int,
               topk_len: Optional[int], cmp_ratio: int = 1, orig_len: Optional[int] = None) -> np.ndarray:
    """Which slots contribute (readings R5, R6).

    A slot is valid iff its key position lies in the sequence (0 <= j < Sk),
    its slot number is below topk_length when that tensor is given (the
    article: topk_length is the number of keys each query row actually
    selected), and, for mask_mode 3, j <= r + Sk - Sq -- with compressed keys
    (R12) the block of key j must end at or before r + L - Sq, L = orig_len.
    """
    L = Sk if orig_len is None else int(orig_len)
    i = np.arange(len(j))
    ok = (j >= 0) & (j < Sk)
    if topk_len is not None:
        ok &= i < int(topk_len)
    if mask_mode == 3:
        ok &= (j + 1) * int(cmp_ratio) - 1 <= (r + L - Sq)
    elif mask_mode != 0:
        raise ValueError("mask_mode must be 0 (none) or 3 (rightDownCausal)")
    return ok


# ----------------------------------------------------------------------------
# stage 2: P = SimpleSoftmax(Mask(Q selectedKv^T scale), softmaxLse)
# ----------------------------------------------------------------------------
def simple_softmax(q_row: np.ndarray, sel_k: np.ndarray, valid: np.ndarray,
                   lse_row: np.ndarray, scale: float) -> np.ndarray:
    """q_row (G, D) and sel_k (n, D) in float64; lse_row (G,).  Returns P (G, n).

    logits = (q_row @ sel_k^T) * scale; masked slots are set to 0 instead of
    exp(-inf - lse) (reading R5); P = exp(logits - lse[g]) (reading R2).
    """
    logits = (q_row @ sel_k.T) * float(scale)
    p = np.zeros_like(logits)
    if valid.any():
        v = np.flatnonzero(valid)
        p[:, v] = np.exp(logits[:, v] - np.asarray(lse_row, dtype=np.float64)[:, None])
    return p


# ----------------------------------------------------------------------------
# stage 3: ReduceSum(P, dimG) / G
# ----------------------------------------------------------------------------
def reduce_sum_g_mean(p: np.ndarray) -> np.ndarray:
    """P (G, n) -> (n,): sum over the head group, divided by G (reading R9)."""
    G = p.shape[0]
    return p.sum(axis=0) / G


# ----------------------------------------------------------------------------
# whole operator
# ----------------------------------------------------------------------------
def _prepare(q_bits, k_bits, dtype, layout, cu_seqlens_q, cu_seqlens_k):
    q_bits = np.asarray(q_bits)
    k_bits = np.asarray(k_bits)
    geo = token_geometry(layout, q_bits.shape, k_bits.shape, cu_seqlens_q, cu_seqlens_k)
    G, D = int(q_bits.shape[-2]), int(q_bits.shape[-1])
    qv = q_bits.reshape(-1, G, D)          # token-major view: (n_tokens, G, D)
    kv = k_bits.reshape(-1, D)             # key rows: (B*S2 or T2, D)
    return geo, G, D, qv, kv


def _width(layout, k_shape, sparse_indices, max_seqlen_k):
    """Output last dimension (reading R3)."""
    if sparse_indices is not None:
        return int(np.asarray(sparse_indices).shape[-1])
    return int(max_seqlen_k) if layout == "TND" else int(k_shape[1])


def _effective(geo_t, seqused_q, seqused_k):
    """(b, r, Sq', k0, Sk') with the participating lengths (reading R11)."""
    b, r, Sq, k0, Sk = geo_t
    if seqused_q is not None:
        Sq = max(0, min(Sq, int(np.asarray(seqused_q).reshape(-1)[b])))
    if seqused_k is not None:
        Sk = max(0, min(Sk, int(np.asarray(seqused_k).reshape(-1)[b])))
    return b, r, Sq, k0, Sk


def original_key_length(Sk: int, b: int, cmp_ratio: int, cmp_residual_k) -> int:
    """L = Sk * c + res of sequence b (reading R12)."""
    c = int(cmp_ratio)
    res = 0 if cmp_residual_k is None else int(np.asarray(cmp_residual_k).reshape(-1)[b])
    return Sk * c + min(max(res, 0), c - 1)


def _row_terms(t, geo, qv, kv, dtype, sparse_indices, topk_length, width, mask_mode,
               seqused_q=None, seqused_k=None, cmp_ratio=1, cmp_residual_k=None):
    b, r, Sq, k0, Sk = _effective(geo[t], seqused_q, seqused_k)
    idx_row = None
    tl = None
    if sparse_indices is not None:
        idx_row = np.asarray(sparse_indices).reshape(len(geo), -1)[t]
        if topk_length is not None:
            tl = int(np.asarray(topk_length).reshape(-1)[t])
    j = slot_key_positions(idx_row, width)
    if int(cmp_ratio) == 1:
        valid = slot_valid(j, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=tl)
    else:
        valid = slot_valid(j, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=tl, cmp_ratio=int(cmp_ratio),
                           orig_len=original_key_length(Sk, b, cmp_ratio, cmp_residual_k))
    if r >= Sq:                                # a query row that does not take part
        valid = np.zeros_like(valid)
    rows = np.where(valid, k0 + j, 0)          # key rows (any row for invalid slots)
    if kv.shape[0] == 0:                       # no key row at all: every slot is invalid
        sel_k = np.zeros((len(rows), kv.shape[1]))
    else:
        sel_k = decode_half(kv[rows], dtype)   # stage 1 gather
    q_row = decode_half(qv[t], dtype)
    return q_row, sel_k, valid


def softmax_l1_norm_rows(q_bits, k_bits, softmax_lse, rows: Iterable[int], *, dtype: str,
                         sparse_indices=None, topk_length=None, cu_seqlens_q=None,
                         cu_seqlens_k=None, softmax_scale: float = 1.0, max_seqlen_k: int = 0,
                         mask_mode: int = 0, layout: str = "BSND", seqused_q=None,
                         seqused_k=None, cmp_ratio: int = 1, cmp_residual_k=None) -> np.ndarray:
    """The operator for selected query tokens only; returns float32 (len(rows), width).

    ``rows`` are token indices (b*S1 + r for BSND, the packed index for TND).
    ``softmax_lse`` is (B,1,S1,G) or (1,T1,G) float32 ([SMLA] 参数说明).
    """
    geo, G, D, qv, kv = _prepare(q_bits, k_bits, dtype, layout, cu_seqlens_q, cu_seqlens_k)
    width = _width(layout, np.asarray(k_bits).shape, sparse_indices, max_seqlen_k)
    lse = np.asarray(softmax_lse, dtype=np.float32).reshape(len(geo), G).astype(np.float64)
    rows = list(rows)
    out = np.zeros((len(rows), width), dtype=np.float32)
    for n, t in enumerate(rows):
        q_row, sel_k, valid = _row_terms(t, geo, qv, kv, dtype, sparse_indices, topk_length,
                                         width, mask_mode, seqused_q, seqused_k, cmp_ratio, cmp_residual_k)
        p = simple_softmax(q_row, sel_k, valid, lse[t], softmax_scale)      # stage 2
        out[n] = reduce_sum_g_mean(p).astype(np.float32)                    # stage 3 (R10)
    return out


def softmax_l1_norm(q_bits, k_bits, softmax_lse, *, dtype: str, sparse_indices=None,
                    topk_length=None, cu_seqlens_q=None, cu_seqlens_k=None,
                    softmax_scale: float = 1.0, max_seqlen_k: int = 0, mask_mode: int = 0,
                    layout: str = "BSND", seqused_q=None, seqused_k=None, cmp_ratio: int = 1,
                    cmp_residual_k=None) -> np.ndarray:
    """The whole operator.  Output float32 (B,S1,1,width) or (T1,1,width)
    ([SMLA] infershape: BSND gives (B, S1, N2, K or S2); TND reading R4)."""
    q_bits = np.asarray(q_bits)
    n_tok = int(np.prod(q_bits.shape[:-2]))
    out = softmax_l1_norm_rows(q_bits, k_bits, softmax_lse, range(n_tok), dtype=dtype,
                               sparse_indices=sparse_indices, topk_length=topk_length,
                               cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                               softmax_scale=softmax_scale, max_seqlen_k=max_seqlen_k,
                               mask_mode=mask_mode, layout=layout, seqused_q=seqused_q,
                               seqused_k=seqused_k, cmp_ratio=cmp_ratio, cmp_residual_k=cmp_residual_k)
    if layout == "TND":
        return out.reshape(n_tok, 1, -1)
    return out.reshape(q_bits.shape[0], q_bits.shape[1], 1, -1)


# ----------------------------------------------------------------------------
# the LSE input, as the forward attention pass defines it
# ----------------------------------------------------------------------------
def softmax_lse(q_bits, k_bits, *, dtype: str, rows: Optional[Iterable[int]] = None,
                sparse_indices=None, topk_length=None, cu_seqlens_q=None, cu_seqlens_k=None,
                softmax_scale: float = 1.0, max_seqlen_k: int = 0, mask_mode: int = 0,
                layout: str = "BSND", seqused_q=None, seqused_k=None, cmp_ratio: int = 1,
                cmp_residual_k=None) -> np.ndarray:
    """softmaxLse of the forward attention pass over the same valid set:
    lse[t, g] = log sum_{valid i} exp(scale * q[t,g] . k[j_i]), float64,
    -inf for a row with no valid slot.  ([SMLA] 参数说明: softmax_lse is the
    forward pass's output; its formula lives in that pass's documentation,
    and this is the log-sum-exp that makes each head's P sum to one.)
    Returns (len(rows), G)."""
    geo, G, D, qv, kv = _prepare(q_bits, k_bits, dtype, layout, cu_seqlens_q, cu_seqlens_k)
    width = _width(layout, np.asarray(k_bits).shape, sparse_indices, max_seqlen_k)
    rows = range(len(geo)) if rows is None else list(rows)
    out = np.full((len(rows), G), -math.inf, dtype=np.float64)
    for n, t in enumerate(rows):
        q_row, sel_k, valid = _row_terms(t, geo, qv, kv, dtype, sparse_indices, topk_length,
                                         width, mask_mode, seqused_q, seqused_k, cmp_ratio, cmp_residual_k)
        if not valid.any():
            continue
        x = (q_row @ sel_k[valid].T) * float(softmax_scale)
        m = x.max(axis=1, keepdims=True)
        out[n] = (m + np.log(np.exp(x - m).sum(axis=1, keepdims=True)))[:, 0]
    return out
