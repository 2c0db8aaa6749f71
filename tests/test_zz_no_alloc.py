"""The allocation-free entry point, smla_l1norm_run_noalloc.

It serves callers that cannot call cudaMalloc (a framework allocator owns
the device memory, a plugin receives pointers but no allocator, a service
forbids allocation after start-up): its work list and status word live in a
fixed device array inside the library instead of a plan's device buffer.

The GPU test calls it through the C ABI twice in a row and compares each
result with the plan-based entry point's, at the tolerance every parity test
here uses.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as W
from smla_harness import (ROWSUM_TOL, assert_close, exact_lse, oracle_kwargs, plan_kwargs, run_gpu,
                          to_device)

import softmax_l1_norm_gb300 as smla


def _desc_kwargs(w):
    kw = plan_kwargs(w)
    return kw


def _call_noalloc(lib, torch, w, t, out):
    d, keep = smla._make_desc(**_desc_kwargs(w))
    code = lib.smla_l1norm_run_noalloc(
        ctypes.byref(d), t["q"].data_ptr(), t["k"].data_ptr(), t["lse"].data_ptr(),
        None if t["idx"] is None else t["idx"].data_ptr(),
        None if t["tl"] is None else t["tl"].data_ptr(), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    del keep
    return code


def test_compressed_keys_under_the_causal_mask_are_not_taken():
    """cmp_residual_k has no argument in the allocation-free entry point, so
    compressed keys with mask_mode 3 are rejected there (before any CUDA
    call); plans take them through smla_l1norm_run_tensors."""
    lib = smla.library()
    d, keep = smla._make_desc(layout="BSND", dtype="bf16", num_heads_q=8, batch_size=1, max_seqlen_q=16,
                              max_seqlen_k=64, topk=8, mask_mode=3, cmp_ratio=4, softmax_scale=1.0)
    assert lib.smla_l1norm_run_noalloc(ctypes.byref(d), None, None, None, None, None, None, None) == \
        smla.SMLA_ERR_UNSUPPORTED
    del keep


def test_capacity_rejected_before_any_cuda_call():
    """More work items than the fixed scratch holds: SMLA_ERR_CAPACITY, with
    no CUDA call (this runs on a host without a GPU)."""
    lib = smla.library()
    d, keep = smla._make_desc(layout="BSND", dtype="bf16", num_heads_q=8, batch_size=2,
                              max_seqlen_q=40000, max_seqlen_k=64, topk=8, softmax_scale=1.0)
    code = lib.smla_l1norm_run_noalloc(ctypes.byref(d), None, None, None, None, None, None, None)
    assert code == smla.SMLA_ERR_CAPACITY
    assert "65536" in lib.smla_status_string(code).decode()
    del keep


OPTIN = 232448  # opt-in shared memory per block of the sm_100 family (227 KB)


@pytest.mark.parametrize("sparse", [True, False])
def test_noalloc_ring_depth_is_even_for_every_head_count(sparse):
    """The launch shape the allocation-free path picks (host query, no GPU):
    for every head count, sparse and dense, the key ring has an even number of
    stages, at least 4, and fits the opt-in shared memory; it is the plan
    path's choice for the same description.  An odd depth would let a barrier
    fall two phases behind with two producer groups."""
    for G in range(1, 129):
        kw = dict(layout="BSND", dtype="bf16", num_heads_q=G, batch_size=1, max_seqlen_q=64,
                  max_seqlen_k=512, topk=256 if sparse else 0, mask_mode=3, softmax_scale=0.05)
        info = smla.noalloc_config(152, OPTIN, **kw)
        assert info.stages % 2 == 0 and 4 <= info.stages <= 12, (G, sparse, info.stages)
        assert info.smem_bytes <= OPTIN
        _, _, plan_info = smla.schedule_host(152, want_items=False, **kw)
        assert (info.stages, info.smem_bytes, info.mma_n, info.rows_per_item) == \
            (plan_info.stages, plan_info.smem_bytes, plan_info.mma_n, plan_info.rows_per_item), G


def test_noalloc_config_counts_items_and_ctas():
    kw = dict(layout="TND", dtype="fp16", num_heads_q=16, batch_size=3, topk=0, mask_mode=3,
              softmax_scale=0.05, cu_seqlens_q=[0, 70, 75, 205], cu_seqlens_k=[0, 90, 95, 225],
              max_seqlen_k=130)
    info = smla.noalloc_config(152, OPTIN, **kw)
    assert info.rows_per_item == 8 and info.num_items == 9 + 1 + 17 and info.num_ctas == 27
    assert info.num_tokens == 205 and info.out_width == 130
    info = smla.noalloc_config(4, OPTIN, **kw)
    assert info.num_ctas == 4
    with pytest.raises(smla.SmlaError) as e:
        smla.noalloc_config(152, OPTIN, layout="BSND", dtype="bf16", num_heads_q=8, batch_size=2,
                            max_seqlen_q=40000, max_seqlen_k=64, topk=8, softmax_scale=1.0)
    assert e.value.code == smla.SMLA_ERR_CAPACITY


@pytest.mark.parametrize("change,code", [
    (dict(num_heads_k=2), smla.SMLA_ERR_INVALID),
    (dict(head_dim=256), smla.SMLA_ERR_INVALID),
    (dict(mask_mode=2), smla.SMLA_ERR_UNSUPPORTED),
    (dict(cmp_ratio=0), smla.SMLA_ERR_INVALID),
    (dict(layout="TND"), smla.SMLA_ERR_NULLPTR),
    (dict(topk=0), smla.SMLA_ERR_INVALID),
])
def test_rejects_like_the_plan_path(change, code):
    lib = smla.library()
    kw = dict(layout="BSND", dtype="bf16", num_heads_q=8, batch_size=1, max_seqlen_q=16,
              max_seqlen_k=256, topk=32, mask_mode=0, softmax_scale=0.044, has_topk_length=True)
    kw.update(change)
    d, keep = smla._make_desc(**kw)
    assert lib.smla_l1norm_run_noalloc(ctypes.byref(d), None, None, None, None, None, None, None) == code
    with pytest.raises(smla.SmlaError) as e:
        smla.Plan(**kw)
    assert e.value.code == code
    del keep


@pytest.mark.gpu
def test_noalloc_matches_plan_path_twice_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = smla.library()
    cases = [
        W.make_workload(name="sparse_causal_G128", layout="BSND", dtype="bf16", B=1, S1=300, S2=1500,
                        G=128, topk=700, mask_mode=3, seed=4100),
        W.make_workload(name="dense_tnd_G16", layout="TND", dtype="fp16", seqlens_q=[70, 5, 130],
                        seqlens_k=[90, 5, 130], G=16, topk=0, mask_mode=3, seed=4101),
    ]
    for w in cases:
        want, plan, t, status = run_gpu(smla, w)
        assert status[0] == smla.SMLA_OK
        d, keep = smla._make_desc(**_desc_kwargs(w))
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):
            out = torch.full(plan.output_shape, float("nan"), dtype=torch.float32, device="cuda")
            code = lib.smla_l1norm_run_noalloc(
                ctypes.byref(d), t["q"].data_ptr(), t["k"].data_ptr(), t["lse"].data_ptr(),
                None if t["idx"] is None else t["idx"].data_ptr(),
                None if t["tl"] is None else t["tl"].data_ptr(), out.data_ptr(), stream)
            assert code == smla.SMLA_OK, lib.smla_status_string(code).decode()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert np.isfinite(got).all(), f"{w.name} call {call}: unwritten elements"
            assert_close(got, want, what=f"{w.name} no-alloc call {call}")
        del keep


@pytest.mark.gpu
@pytest.mark.parametrize("G,topk,layout", [(40, 300, "BSND"), (72, 300, "BSND"), (100, 300, "BSND"),
                                           (33, 0, "BSND"), (56, 0, "TND")])
def test_noalloc_matches_the_oracle_at_every_ring_depth(G, topk, layout):
    """Head counts whose shared-memory footprint leaves room for an odd number
    of key stages (G 33-48, 65-80, 97-112 sparse; dense packs of R*G in the
    same ranges): the allocation-free path takes the plan path's even depth,
    and its output equals the oracle's element by element, twice in a row."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = smla.library()
    if layout == "BSND":
        w = W.make_workload(layout="BSND", dtype="bf16" if topk else "fp16", B=2, S1=21, S2=700, G=G,
                            topk=topk, mask_mode=3, seed=4200 + G, lse=None)
    else:
        w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[40, 3, 90], seqlens_k=[60, 3, 300],
                            G=G, topk=topk, mask_mode=3, seed=4200 + G, lse=None)
    exact_lse(oracle, w)
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    info = smla.noalloc_config(torch.cuda.get_device_properties(0).multi_processor_count,
                               232448, **_desc_kwargs(w))
    assert info.stages % 2 == 0 and info.stages >= 4
    t = to_device(w)
    for call in range(2):
        out = torch.full(want.shape, float("nan"), dtype=torch.float32, device="cuda")
        code = _call_noalloc(lib, torch, w, t, out)
        assert code == smla.SMLA_OK, lib.smla_status_string(code).decode()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert_close(got, want, what=f"G={G} topk={topk} {layout} no-alloc call {call}")
        rows = got.reshape(w.n_tokens, -1).astype(np.float64)
        has = ~np.isneginf(w.lse_rows()[:, 0])
        assert np.all(np.abs(rows[has].sum(axis=1) - 1.0) <= ROWSUM_TOL)


@pytest.mark.gpu
def test_noalloc_after_plans_of_other_footprints():
    """A large-footprint plan, a small one, the large one again, then the
    allocation-free path at a third footprint: creating a plan never lowers
    the shared-memory cap another launch relies on."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lib = smla.library()
    big = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=12, S2=600, G=128, topk=256, mask_mode=3,
                          seed=4300, lse=None)
    small = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=12, S2=600, G=8, topk=256, mask_mode=3,
                            seed=4301, lse=None)
    mid = W.make_workload(layout="BSND", dtype="fp16", B=1, S1=30, S2=300, G=16, topk=0, mask_mode=3,
                          seed=4302, lse=None)
    for w in (big, small, mid):
        exact_lse(oracle, w)
    want = {id(w): oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
            for w in (big, small, mid)}
    got_big, plan_big, t_big, st = run_gpu(smla, big)
    assert st[0] == smla.SMLA_OK
    assert_close(got_big, want[id(big)], what="G=128 plan")
    got_small, plan_small, _, st = run_gpu(smla, small)
    assert st[0] == smla.SMLA_OK and plan_small.info.smem_bytes < plan_big.info.smem_bytes
    assert_close(got_small, want[id(small)], what="G=8 plan")
    again, _, _, st = run_gpu(smla, big, plan=plan_big, tensors=t_big)
    assert st[0] == smla.SMLA_OK
    assert_close(again, want[id(big)], what="G=128 plan after the G=8 plan")
    t = to_device(mid)
    out = torch.full(want[id(mid)].shape, float("nan"), dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, torch, mid, t, out) == smla.SMLA_OK
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), want[id(mid)], what="dense G=16 no-alloc after both plans")
