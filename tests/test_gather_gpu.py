"""Stage 1 of the operator (article "SparseFlashMlaSoftmaxL1Norm", section
三阶段计算公式: selectedKv = Gather(K, sparse_indices)), checked bit for bit.

``smla_debug_gather`` runs the key-producer warps of the fused kernel -- the
same device code -- for one work item, with a stand-in for the tensor cores
that copies every shared-memory ring stage out exactly as the MMA reads it.
Each stage is compared byte for byte with the key rows the slots name,
placed by the definition of the 128-byte swizzle (16-byte piece p of row s
of an 8-row group at position p XOR (s mod 8)).  Invalid slots (index -1,
out of range, past topk_length or topk, past the sequence's keys) must hold
zeros: nothing is read for them, and the epilogue masks them.
"""
import numpy as np
import pytest

import workloads as W
from smla_harness import plan_kwargs, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

STAGE = 16384
SENTINEL = 0xA5


def item_of(w, R, token):
    """(first local row, rows) of the work item holding ``token``."""
    b, r, Sq, k0, Sk = (int(x) for x in w.token_table()[token])
    r0 = (r // R) * R
    return r0, min(R, Sq - r0)


def expected_stages(w, token, R):
    """The ring stages of the item holding ``token``, as bytes (stages, 128, 128)."""
    b, r, Sq, k0, Sk = (int(x) for x in w.token_table()[token])
    keys = np.ascontiguousarray(w.k_bits.reshape(-1, 512)).view(np.uint8)   # 1024 bytes per key row
    if w.sparse_indices is not None:
        topk = w.topk
        tl = topk if w.topk_length is None else min(max(int(w.topk_length.reshape(-1)[token]), 0), topk)
        if Sk == 0:
            tl = 0
        ntiles = -(-tl // 128)
        idx = w.sparse_indices.reshape(w.n_tokens, -1)[token].astype(np.int64)
        slots = np.arange(ntiles * 128)
        j = np.where(slots < tl, idx[np.minimum(slots, topk - 1)], -1)
    else:
        r0, nrows = item_of(w, R, token)
        last = r0 + nrows - 1
        vis = Sk if w.mask_mode == 0 else min(Sk, max(0, last + Sk - Sq + 1))
        ntiles = -(-min(vis, w.out_width) // 128)
        j = np.arange(ntiles * 128)
    valid = (j >= 0) & (j < Sk)
    gathered = keys[k0 + np.where(valid, j, 0)].copy()
    gathered[~valid] = 0   # invalid slots are zero-filled
    src = gathered.reshape(ntiles, 128, 8, 8, 16).transpose(0, 2, 1, 3, 4)  # tile, chunk, slot, piece, byte
    # position q of slot s holds piece q XOR (s mod 8)
    piece_at = np.arange(8)[None, :] ^ (np.arange(128)[:, None] & 7)
    out = np.take_along_axis(src, piece_at[None, None, :, :, None], axis=3)
    return np.ascontiguousarray(out).reshape(ntiles * 8, 128, 128)


def check_gather(lib, w, tokens, modes=(0, 1), **plan_extra):
    plan = lib.Plan(**plan_kwargs(w, **plan_extra))
    R = plan.info.rows_per_item
    t = to_device(w)
    for token in tokens:
        want = expected_stages(w, token, R)
        for mode in modes:
            n_stages = want.shape[0] + 2   # two spare stages must stay untouched
            dump = torch.full((n_stages * STAGE,), SENTINEL, dtype=torch.uint8, device="cuda")
            plan.debug_gather(token, t["k"], dump, sparse_indices=t["idx"], topk_length=t["tl"], mode=mode)
            torch.cuda.synchronize()
            got = dump.cpu().numpy().reshape(n_stages, 128, 128)
            assert np.all(got[want.shape[0]:] == SENTINEL), f"token {token} mode {mode}: stages past the item"
            bad = np.argwhere(got[:want.shape[0]] != want)
            assert bad.size == 0, (f"token {token} mode {mode}: {len(bad)} bytes differ, first "
                                   f"(stage, slot, byte) {bad[:4].tolist()}")
    return plan


def test_gather_sparse_padding_and_ragged_tail(lib):
    """Causal top-300 (a ragged third tile), topk_length below topk on early
    rows with -1 padding after it, G = 128 (6-stage ring)."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=40, S2=300, G=128, topk=300, mask_mode=3,
                        seed=5100)
    tl = w.topk_length.reshape(-1)
    tokens = [0, 5, int(np.argmin(tl)), 39]
    check_gather(lib, w, tokens)


def test_gather_out_of_range_indices_without_topk_length(lib):
    """No topk_length: every slot is a candidate; indices below -1 or past Sk
    give zero rows (and raise the bad-index flag)."""
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=6, S2=300, G=16, topk=200, mask_mode=0,
                        seed=5101, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(5101))
    w.sparse_indices = rng.integers(-3, 330, size=w.sparse_indices.shape).astype(np.int32)
    plan = check_gather(lib, w, [0, 7, 11])
    code, flags = plan.status()
    assert code == lib.SMLA_WARN_BAD_INDEX and (flags & 1)


def test_gather_tnd_key_offsets(lib):
    """TND: a slot's key row is cu_seqlens_k[b] + j; tokens of the second and
    third sequence read their own keys.  G = 64 (10-stage ring), topk 1001."""
    w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[30, 45, 20], seqlens_k=[600, 1300, 40],
                        G=64, topk=1001, mask_mode=0, seed=5102)
    check_gather(lib, w, [3, 30 + 44, 75 + 19])


def test_gather_dense_items(lib):
    """Dense form: a pack of R = 128 // G tokens gathers keys 0.. of its
    sequence in order, up to the last row's causal limit."""
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=300, S2=450, G=16, topk=0, mask_mode=3,
                        seed=5103)
    check_gather(lib, w, [0, 13, 299, 300 + 170])


def test_gather_small_head_count_deep_ring(lib):
    """G = 8: the q block is small and the ring takes 12 stages."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=8, S2=4000, G=8, topk=2048, mask_mode=0,
                        seed=5104)
    plan = check_gather(lib, w, [0, 7])
    assert plan.info.stages == 12
