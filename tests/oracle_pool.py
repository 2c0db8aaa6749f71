"""The oracle over many rows at once, spread over host processes.

Test infrastructure: each worker runs the oracle's own functions, unchanged,
on a share of the rows (the exact forward LSE of a row, then the operator's
row from that LSE rounded to fp32, as the GPU receives it).  Workers are
started with ``spawn`` (safe after the parent has initialised CUDA), read the
workload arrays through read-only memory maps of .npy files the parent wrote,
and run one BLAS thread each.
"""
from __future__ import annotations

import json
import multiprocessing as mp
import os

import numpy as np

_ARRAYS = ("q_bits", "k_bits", "sparse_indices", "topk_length", "cu_seqlens_q", "cu_seqlens_k")
_STATE = {}


def _init(folder):
    import oracle
    with open(os.path.join(folder, "meta.json")) as f:
        meta = json.load(f)
    arr = {}
    for name in _ARRAYS:
        path = os.path.join(folder, name + ".npy")
        arr[name] = np.load(path, mmap_mode="r") if os.path.exists(path) else None
    _STATE.update(oracle=oracle, meta=meta, arr=arr)


def _kwargs():
    a, m = _STATE["arr"], _STATE["meta"]
    return dict(dtype=m["dtype"], sparse_indices=a["sparse_indices"], topk_length=a["topk_length"],
                cu_seqlens_q=a["cu_seqlens_q"], cu_seqlens_k=a["cu_seqlens_k"],
                softmax_scale=m["softmax_scale"], max_seqlen_k=m["max_seqlen_k"], mask_mode=m["mask_mode"],
                layout=m["layout"])


def _rows(chunk):
    oracle, a, m = _STATE["oracle"], _STATE["arr"], _STATE["meta"]
    kw = _kwargs()
    lse = oracle.softmax_lse(a["q_bits"], a["k_bits"], rows=chunk, **kw).astype(np.float32)
    full = np.zeros((m["n_tokens"], m["G"]), np.float32)
    full[chunk] = lse
    out = oracle.softmax_l1_norm_rows(a["q_bits"], a["k_bits"], full, chunk, **kw)
    return chunk, lse, out


def lse_and_rows(w, rows, folder, processes=None, chunk=16):
    """Exact forward LSE (fp32) and the operator's output for ``rows`` of
    workload ``w``, in row order.  ``folder`` receives the memory-mapped
    copies of the inputs."""
    rows = list(rows)
    os.makedirs(folder, exist_ok=True)
    for name in _ARRAYS:
        v = getattr(w, name)
        if v is not None:
            np.save(os.path.join(folder, name + ".npy"), np.ascontiguousarray(v))
    meta = dict(dtype=w.dtype, softmax_scale=float(w.softmax_scale), max_seqlen_k=int(w.max_seqlen_k),
                mask_mode=int(w.mask_mode), layout=w.layout, n_tokens=int(w.n_tokens), G=int(w.G))
    with open(os.path.join(folder, "meta.json"), "w") as f:
        json.dump(meta, f)
    procs = processes or max(1, min(len(os.sched_getaffinity(0)), 32))
    chunks = [rows[i:i + chunk] for i in range(0, len(rows), chunk)]
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for v in saved:
        os.environ[v] = "1"
    try:
        with mp.get_context("spawn").Pool(procs, initializer=_init, initargs=(folder,)) as pool:
            parts = pool.map(_rows, chunks)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    lse = np.concatenate([p[1] for p in parts]) if parts else np.zeros((0, w.G), np.float32)
    out = np.concatenate([p[2] for p in parts]) if parts else np.zeros((0, w.out_width), np.float32)
    return lse, out
