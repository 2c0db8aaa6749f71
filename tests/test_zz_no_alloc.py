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

import workloads as W
from smla_harness import assert_close, plan_kwargs, run_gpu, to_device

import softmax_l1_norm_gb300 as smla


def _desc_kwargs(w):
    kw = plan_kwargs(w)
    return kw


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


@pytest.mark.parametrize("change,code", [
    (dict(num_heads_k=2), smla.SMLA_ERR_INVALID),
    (dict(head_dim=256), smla.SMLA_ERR_INVALID),
    (dict(mask_mode=2), smla.SMLA_ERR_UNSUPPORTED),
    (dict(cmp_ratio=4), smla.SMLA_ERR_UNSUPPORTED),
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
