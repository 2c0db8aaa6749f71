"""The C-ABI library on the host (no GPU): it builds, loads, exports every
symbol the header declares, rejects bad descriptions before any CUDA call,
and its scheduler covers every query token exactly once with a balanced load."""
import ctypes
import os
import re

import numpy as np
import pytest

import softmax_l1_norm_gb300 as smla
import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "smla_l1norm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(smla_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for must in ("smla_l1norm_plan_create", "smla_l1norm_run", "smla_l1norm_plan_destroy",
                 "smla_l1norm_output_shape", "smla_l1norm_get_status", "smla_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(smla.library_path() if os.path.exists(smla.library_path()) else smla.library()._name)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings():
    lib = smla.library()
    for code in range(7):
        s = lib.smla_status_string(code).decode()
        assert s.startswith("SMLA_")
    assert "unknown" in lib.smla_status_string(99).decode()


BASE = dict(layout="BSND", dtype="bf16", num_heads_q=8, batch_size=1, max_seqlen_q=16,
            max_seqlen_k=256, topk=32, mask_mode=0, softmax_scale=0.044, has_topk_length=True)


@pytest.mark.parametrize("change,code", [
    (dict(num_heads_k=2), smla.SMLA_ERR_INVALID),          # N2 only 1
    (dict(num_heads_q=0), smla.SMLA_ERR_INVALID),
    (dict(num_heads_q=129), smla.SMLA_ERR_INVALID),        # N1 in 1..128
    (dict(head_dim=256), smla.SMLA_ERR_INVALID),           # D only 512
    (dict(mask_mode=2), smla.SMLA_ERR_UNSUPPORTED),
    (dict(mask_mode=5), smla.SMLA_ERR_INVALID),
    (dict(cmp_ratio=0), smla.SMLA_ERR_INVALID),
    (dict(cmp_ratio=129), smla.SMLA_ERR_INVALID),
    (dict(dtype=7), smla.SMLA_ERR_INVALID),
    (dict(topk=-1), smla.SMLA_ERR_INVALID),
    (dict(topk=0), smla.SMLA_ERR_INVALID),                 # topk_length without indices
    (dict(batch_size=-1), smla.SMLA_ERR_INVALID),
    (dict(softmax_scale=float("nan")), smla.SMLA_ERR_INVALID),
    (dict(layout="TND"), smla.SMLA_ERR_NULLPTR),           # TND needs cu_seqlens
    (dict(layout="TND", cu_seqlens_q=[0, 4, 2], cu_seqlens_k=[0, 4, 8], batch_size=2), smla.SMLA_ERR_INVALID),
    (dict(layout="TND", cu_seqlens_q=[1, 4], cu_seqlens_k=[0, 4], batch_size=1), smla.SMLA_ERR_INVALID),
    (dict(layout="TND", topk=0, has_topk_length=False, cu_seqlens_q=[0, 4], cu_seqlens_k=[0, 9],
          batch_size=1, max_seqlen_k=8), smla.SMLA_ERR_INVALID),   # width below a sequence's length
])
def test_plan_rejects_before_any_cuda_call(change, code):
    kw = {**BASE, **change}
    with pytest.raises(smla.SmlaError) as e:
        smla.Plan(**kw)
    assert e.value.code == code


def test_layout_mismatch_and_null_desc():
    lib = smla.library()
    d, keep = smla._make_desc(**BASE)
    d.layout_k = 1
    h = ctypes.c_void_p()
    assert lib.smla_l1norm_plan_create(ctypes.byref(d), ctypes.byref(h)) == smla.SMLA_ERR_INVALID
    assert lib.smla_l1norm_plan_create(None, ctypes.byref(h)) == smla.SMLA_ERR_NULLPTR
    d.layout_k = 0
    assert lib.smla_l1norm_plan_create(ctypes.byref(d), None) == smla.SMLA_ERR_NULLPTR
    assert lib.smla_l1norm_run(None, None, None, None, None, None, None, None) == smla.SMLA_ERR_NULLPTR
    assert lib.smla_l1norm_run_tensors(None, None, None) == smla.SMLA_ERR_NULLPTR


def _tokens_of(items):
    seen = []
    for it in items:
        q_tok, nrows = it[0], it[1]
        seen.extend(range(q_tok, q_tok + nrows))
    return seen


@pytest.mark.parametrize("G,topk,mask,layout", [
    (128, 2048, 3, "BSND"), (8, 32, 0, "BSND"), (16, 0, 3, "BSND"), (64, 2048, 3, "TND"),
    (1, 0, 0, "TND"), (3, 0, 3, "BSND"), (24, 300, 3, "TND")])
def test_schedule_covers_every_token_once(G, topk, mask, layout):
    if layout == "TND":
        lens = [7, 300, 0, 129, 1000]
        cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
        kw = dict(layout="TND", cu_seqlens_q=cu, cu_seqlens_k=cu, batch_size=len(lens),
                  max_seqlen_k=max(lens))
        n_tok = cu[-1]
    else:
        kw = dict(layout="BSND", batch_size=2, max_seqlen_q=700, max_seqlen_k=900)
        n_tok = 1400
    items, offs, info = smla.schedule_host(97, num_heads_q=G, topk=topk, mask_mode=mask,
                                           has_topk_length=topk > 0, softmax_scale=0.05, **kw)
    assert offs[0] == 0 and offs[-1] == len(items) == info.num_items
    assert all(a <= b for a, b in zip(offs, offs[1:]))
    toks = _tokens_of(items)
    assert sorted(toks) == list(range(n_tok))
    # the last field is the item's sequence number (it indexes seqused_q / seqused_k)
    if layout == "TND":
        for it in items:
            b = it[7]
            assert cu[b] <= it[0] < cu[b + 1] and it[3] == cu[b]
    else:
        assert all(it[7] == it[0] // 700 for it in items)
    if topk > 0:
        assert info.rows_per_item == 1 and info.mma_n == max(16, -(-G // 16) * 16)
    else:
        assert info.rows_per_item == max(1, 128 // G)
        assert info.mma_n <= 128
    assert info.smem_bytes <= 232448 and 4 <= info.stages <= 12


@pytest.mark.parametrize("topk", [256, 0])
def test_key_ring_depth_is_even_for_every_head_count(topk):
    """The key ring always has an even number of stages, at least 4: with two
    producer groups filling alternate stages, an odd depth would let an MMA
    issuer test a stage's full barrier two phases early.  Sparse and dense."""
    for G in range(1, 129):
        _, _, info = smla.schedule_host(152, want_items=False, num_heads_q=G, batch_size=1,
                                        max_seqlen_q=64, max_seqlen_k=512, topk=topk, mask_mode=3,
                                        has_topk_length=False, softmax_scale=0.05)
        assert info.stages % 2 == 0 and 4 <= info.stages <= 12, (G, info.stages)
        assert info.smem_bytes <= 232448


def test_compressed_keys_are_accepted_and_bound_the_dense_tiles():
    """cmp_ratio 2..128 is accepted.  The host does not see cmp_residual_k
    (a device tensor), so dense work items are sized for the largest
    residual, c - 1: key j of row r counts when j*c + c - 1 <= r + Sk*c + c - 1 - Sq."""
    S1, Sk, c = 64, 40, 8
    items, _, info = smla.schedule_host(4, num_heads_q=16, batch_size=1, max_seqlen_q=S1, max_seqlen_k=Sk,
                                        topk=0, mask_mode=3, softmax_scale=0.05, cmp_ratio=c)
    assert info.out_width == Sk
    for q_tok, nrows, r0, k_base, Sq, Sk_, ntiles, *_ in items:
        last = r0 + nrows - 1
        vis = min(Sk, max(0, last + Sk * c + (c - 1) - S1 + 1) // c)
        assert ntiles == -(-vis // 128)
    _, _, info = smla.schedule_host(4, want_items=False, num_heads_q=8, batch_size=1, max_seqlen_q=16,
                                    max_seqlen_k=300, topk=64, mask_mode=3, softmax_scale=0.05, cmp_ratio=128,
                                    has_topk_length=True)
    assert info.num_items == 16


def test_mma_issuers_follow_the_accumulator_width():
    """The sparse L1-norm launch uses four MMA issuers when each one's
    accumulator (the MMA N, G padded to 16) fits in a quarter of a 256-column
    TMEM buffer; the dense form and wider sparse N use two."""
    for G in (1, 16, 48, 64, 65, 80, 128):
        _, _, info = smla.schedule_host(152, want_items=False, num_heads_q=G, batch_size=1, max_seqlen_q=8,
                                        max_seqlen_k=512, topk=256, mask_mode=0, softmax_scale=0.05)
        assert info.mma_issuers == (4 if info.mma_n <= 64 else 2), (G, info.mma_n, info.mma_issuers)
        nf = smla.noalloc_config(152, 232448, num_heads_q=G, batch_size=1, max_seqlen_q=8,
                                 max_seqlen_k=512, topk=256, mask_mode=0, softmax_scale=0.05)
        assert nf.mma_issuers == info.mma_issuers
    _, _, info = smla.schedule_host(152, want_items=False, num_heads_q=16, batch_size=1, max_seqlen_q=64,
                                    max_seqlen_k=512, topk=0, mask_mode=3, softmax_scale=0.05)
    assert info.mma_issuers == 2


def test_schedule_balance_on_the_causal_topk2048_shape():
    """4096 tokens, G=128, topk 2048 causal: per-token work runs from 1 to 16
    tiles; longest-first assignment keeps the heaviest CTA within a few % of
    the mean."""
    _, _, info = smla.schedule_host(152, want_items=False, num_heads_q=128, batch_size=1,
                                    max_seqlen_q=4096, max_seqlen_k=4096, topk=2048, mask_mode=3,
                                    has_topk_length=True, softmax_scale=0.044)
    assert info.num_items == 4096
    tiles = sum(-(-min(2048, i + 1) // 128) for i in range(4096))
    assert info.est_tiles == tiles
    assert info.max_cta_cost <= 1.03 * info.mean_cta_cost


def test_topk_length_hint_drives_the_estimate():
    hint = [5] * 16
    _, _, info = smla.schedule_host(4, want_items=False, num_heads_q=8, batch_size=1, max_seqlen_q=16,
                                    max_seqlen_k=4096, topk=2048, mask_mode=0, has_topk_length=True,
                                    softmax_scale=1.0, topk_length_hint=hint)
    assert info.est_tiles == 16


def test_dense_items_respect_causal_visibility():
    items, _, _ = smla.schedule_host(8, num_heads_q=16, batch_size=1, max_seqlen_q=512,
                                     max_seqlen_k=512, topk=0, mask_mode=3, softmax_scale=0.05)
    for q_tok, nrows, r0, k_base, Sq, Sk, ntiles, *_ in items:
        last = r0 + nrows - 1
        assert ntiles == -(-min(512, last + 1) // 128)


# ---------------------------------------------------------------- dense key split
def _split_cover(items, width):
    """(token pack, key tile) -> count over the items, and the tail writers."""
    cover, tails = {}, {}
    for q_tok, nrows, r0, k_base, Sq, Sk, ntiles, b, t0, cut, r1, r2 in items:
        assert r1 == 0 and r2 == 0 and t0 >= 0 and ntiles >= 0 and cut in (0, 1)
        for t in range(t0, t0 + ntiles):
            cover[(q_tok, t)] = cover.get((q_tok, t), 0) + 1
        if cut == 0:
            tails[q_tok] = tails.get(q_tok, 0) + 1
    return cover, tails


@pytest.mark.parametrize("split", [1, 2, 3, 5])
@pytest.mark.parametrize("layout", ["BSND", "TND"])
def test_dense_split_covers_every_key_tile_once(split, layout):
    """Split into parts of at most ``split`` key tiles, the dense schedule
    covers each (token pack, key tile) of the whole-pack schedule exactly
    once, parts of a pack are contiguous from tile 0, and exactly one part of
    each pack (the last) zeroes the row past its tiles."""
    if layout == "TND":
        lens_q, lens_k = [7, 300, 0, 129, 700], [9, 513, 3, 129, 640]
        kw = dict(layout="TND", cu_seqlens_q=np.concatenate([[0], np.cumsum(lens_q)]).tolist(),
                  cu_seqlens_k=np.concatenate([[0], np.cumsum(lens_k)]).tolist(), batch_size=5,
                  max_seqlen_k=max(lens_k))
    else:
        kw = dict(layout="BSND", batch_size=2, max_seqlen_q=700, max_seqlen_k=900)
    for mask in (0, 3):
        whole, _, _ = smla.schedule_host(37, num_heads_q=16, topk=0, mask_mode=mask, softmax_scale=0.05, **kw)
        parts, offs, info = smla.schedule_host(37, split_tiles=split, num_heads_q=16, topk=0, mask_mode=mask,
                                               softmax_scale=0.05, **kw)
        assert info.split_tiles == split and info.split_items == len(parts) == offs[-1]
        want = {(it[0], t): 1 for it in whole for t in range(it[6])}
        cover, tails = _split_cover(parts, info.out_width)
        assert cover == want
        assert sorted(tails) == sorted(it[0] for it in whole) and set(tails.values()) == {1}
        assert all(it[6] <= split for it in parts)
        # the tail part is the pack's last: no part of the pack starts after it
        last_t0 = {}
        for it in parts:
            last_t0[it[0]] = max(last_t0.get(it[0], 0), it[8])
        assert all(it[8] == last_t0[it[0]] for it in parts if it[9] == 0)


def test_dense_split_choice():
    """The dense L1-norm launch splits a few long packs (2 x 512 causal
    tokens of 16 heads: 128 packs of up to 4 tiles for 152 CTAs) and leaves a
    schedule that is already balanced alone; the sparse form never splits."""
    _, _, info = smla.schedule_host(152, want_items=False, split_tiles=-1, num_heads_q=16, batch_size=2,
                                    max_seqlen_q=512, max_seqlen_k=512, topk=0, mask_mode=3, softmax_scale=0.05)
    assert 0 < info.split_tiles < 4 and info.split_items > 128
    whole = smla.schedule_host(152, want_items=False, num_heads_q=16, batch_size=2, max_seqlen_q=512,
                               max_seqlen_k=512, topk=0, mask_mode=3, softmax_scale=0.05)[2]
    assert info.max_cta_cost < 0.9 * whole.max_cta_cost
    _, _, info = smla.schedule_host(152, want_items=False, split_tiles=-1, num_heads_q=16, batch_size=8,
                                    max_seqlen_q=4096, max_seqlen_k=4096, topk=0, mask_mode=0, softmax_scale=0.05)
    assert info.split_tiles == 0 and info.split_items == 0
    _, _, info = smla.schedule_host(152, want_items=False, split_tiles=-1, num_heads_q=128, batch_size=1,
                                    max_seqlen_q=64, max_seqlen_k=4096, topk=2048, mask_mode=3, softmax_scale=0.05)
    assert info.split_tiles == 0
    with pytest.raises(smla.SmlaError):
        smla.schedule_host(152, want_items=False, split_tiles=2, num_heads_q=128, batch_size=1, max_seqlen_q=64,
                           max_seqlen_k=4096, topk=2048, mask_mode=3, softmax_scale=0.05)
