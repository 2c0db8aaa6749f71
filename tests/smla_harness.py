"""Shared helpers: build plans from a seeded workload and run the CUDA
library on it; compare with the oracle at the operator's tolerance."""
from __future__ import annotations

import numpy as np

# |gpu - oracle| <= ATOL + RTOL * |oracle| per element; row sums within 1e-3 of 1
ATOL = 1e-5
RTOL = 2e-3
ROWSUM_TOL = 1e-3


def plan_kwargs(w, **extra):
    kw = dict(layout=w.layout, dtype=w.dtype, num_heads_q=w.G, batch_size=w.batch,
              max_seqlen_q=w.max_seqlen_q if w.layout == "BSND" else 0,
              max_seqlen_k=(w.k_bits.shape[1] if w.layout == "BSND" else w.max_seqlen_k),
              topk=w.topk, mask_mode=w.mask_mode, softmax_scale=w.softmax_scale,
              has_topk_length=w.topk_length is not None,
              cu_seqlens_q=None if w.cu_seqlens_q is None else w.cu_seqlens_q.tolist(),
              cu_seqlens_k=None if w.cu_seqlens_k is None else w.cu_seqlens_k.tolist())
    kw.update(extra)
    return kw


def to_device(w, device="cuda"):
    import torch
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    t = {}
    t["q"] = torch.from_numpy(w.q_bits.view(np.int16)).view(tdt).to(device)
    t["k"] = torch.from_numpy(w.k_bits.view(np.int16)).view(tdt).to(device)
    t["lse"] = torch.from_numpy(np.ascontiguousarray(w.softmax_lse, dtype=np.float32)).to(device)
    t["idx"] = None if w.sparse_indices is None else torch.from_numpy(
        np.ascontiguousarray(w.sparse_indices, dtype=np.int32)).to(device)
    t["tl"] = None if w.topk_length is None else torch.from_numpy(
        np.ascontiguousarray(w.topk_length, dtype=np.int32)).to(device)
    return t


def run_gpu(smla, w, plan=None, tensors=None, **plan_extra):
    """Run the library on workload ``w``; returns (out numpy, plan, tensors, status)."""
    import torch
    plan = plan or smla.Plan(**plan_kwargs(w, **plan_extra))
    t = tensors or to_device(w)
    out = plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"])
    torch.cuda.synchronize()
    status = plan.status()
    return out.cpu().numpy(), plan, t, status


def oracle_kwargs(w):
    return dict(dtype=w.dtype, sparse_indices=w.sparse_indices, topk_length=w.topk_length,
                cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k,
                softmax_scale=w.softmax_scale, max_seqlen_k=w.max_seqlen_k,
                mask_mode=w.mask_mode, layout=w.layout)


def exact_lse(oracle, w, rows=None):
    """Replace softmax_lse (all rows, or only ``rows``) with the oracle's exact
    forward LSE over the valid set."""
    import workloads as W
    lse_rows = w.lse_rows().copy() if w.softmax_lse is not None else np.zeros((w.n_tokens, w.G), np.float32)
    sel = range(w.n_tokens) if rows is None else rows
    vals = oracle.softmax_lse(w.q_bits, w.k_bits, rows=sel, **oracle_kwargs(w))
    lse_rows[list(sel)] = vals.astype(np.float32)
    W.set_lse_rows(w, lse_rows)
    return w


def assert_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    err = np.abs(got - want)
    bad = ~(err <= ATOL + RTOL * np.abs(want))
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"max err {err.max():.3e}; first {i.tolist()} got "
                             f"{got[tuple(i.T)]} want {want[tuple(i.T)]}")


def invalid_slot_mask(w):
    """Slots that must be exactly 0 whatever the values: past topk_length, or
    with an index outside the sequence (sparse); past the sequence or hidden by
    the causal mask (dense).  Returns bool (n_tokens, width)."""
    tab = w.token_table()
    width = w.out_width
    if w.sparse_indices is not None:
        idx = w.sparse_indices.reshape(w.n_tokens, -1).astype(np.int64)
        Sk = tab[:, 4:5]
        bad = (idx < 0) | (idx >= Sk)
        if w.mask_mode == 3:
            bad |= idx > (tab[:, 1:2] + Sk - tab[:, 2:3])
        if w.topk_length is not None:
            bad |= np.arange(width)[None, :] >= w.topk_length.reshape(-1, 1)
        return bad
    j = np.arange(width)[None, :]
    Sk = tab[:, 4:5]
    bad = j >= Sk
    if w.mask_mode == 3:
        bad |= j > (tab[:, 1:2] + Sk - tab[:, 2:3])
    return bad
