"""GPU parity of the forward-LSE modes (smla_softmax_lse_run and
smla_l1norm_run_fused_lse) against the fp64 oracle, through the C ABI.

Tolerance on the LSE: |gpu - oracle| <= 1e-4 + 1e-6 |oracle|, and -inf
exactly where the oracle has -inf (a row with no kept slot).  The bound
comes from the operator's own tolerance: an LSE error d scales every output
of its row by exp(-d), so d <= 1e-4 keeps the L1-norm output 20x inside its
2e-3 relative bound.  The arithmetic gives about 1e-5 at most: the logits
carry the tensor-core fp32 accumulation error (~1e-6 at scale 1/sqrt(512)),
each exp2 term 2 ulp, the fp32 running sum over up to 2048 terms a few 1e-6
relative.  The fused mode's L1-norm output is held to the operator's
tolerance against the oracle run with the oracle's own LSE, and its rows
must sum to 1."""
import numpy as np
import pytest

import oracle
import workloads as W
from smla_harness import ROWSUM_TOL, assert_close, oracle_kwargs, plan_kwargs, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

LSE_ATOL = 1e-4
LSE_RTOL = 1e-6


def assert_lse_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    ninf_w, ninf_g = np.isneginf(want), np.isneginf(got)
    assert np.array_equal(ninf_w, ninf_g), f"{what}: -inf rows differ ({ninf_w.sum()} vs {ninf_g.sum()})"
    fin = ~ninf_w
    assert np.all(np.isfinite(got[fin])), f"{what}: non-finite LSE"
    err = np.abs(got[fin] - want[fin])
    bad = err > LSE_ATOL + LSE_RTOL * np.abs(want[fin])
    assert not bad.any(), f"{what}: {bad.sum()} LSE values out of tolerance, max err {err.max():.3e}"


def _dev_i32(v):
    return None if v is None else torch.tensor(np.asarray(v, np.int32), device="cuda")


def lse_parity(lib, w, su_q=None, su_k=None, expect=None, rows=None):
    """LSE-only and fused modes on workload ``w``; ``rows`` limits the oracle
    comparison to a sample of tokens (full-size cases)."""
    kw = oracle_kwargs(w)
    kw.update(seqused_q=su_q, seqused_k=su_k)
    sel = list(range(w.n_tokens)) if rows is None else list(rows)
    want_lse = oracle.softmax_lse(w.q_bits, w.k_bits, rows=sel, **kw)
    if w.softmax_lse is None:  # the modes under test do not read it
        W.set_lse_rows(w, np.zeros((w.n_tokens, w.G), np.float32))
    plan = lib.Plan(**plan_kwargs(w))
    t = to_device(w)
    extra = dict(sparse_indices=t["idx"], topk_length=t["tl"], seqused_q=_dev_i32(su_q),
                 seqused_k=_dev_i32(su_k))
    lse = plan.softmax_lse(t["q"], t["k"], **extra)
    torch.cuda.synchronize()
    code, _ = plan.status()
    assert code == (lib.SMLA_OK if expect is None else expect)
    assert tuple(lse.shape) == tuple(w.softmax_lse.shape) == plan.lse_shape
    lse_rows = lse.cpu().numpy().reshape(w.n_tokens, w.G)
    assert_lse_close(lse_rows[sel], want_lse, what=f"{w.name} lse")

    out, lse_f = plan.run_fused_lse(t["q"], t["k"], **extra)
    torch.cuda.synchronize()
    code, _ = plan.status()
    assert code == (lib.SMLA_OK if expect is None else expect)
    # the fused launch runs the same LSE pass
    assert np.array_equal(lse_f.cpu().numpy().reshape(w.n_tokens, w.G).view(np.uint32), lse_rows.view(np.uint32))
    full = w.lse_rows().copy()
    full[sel] = want_lse.astype(np.float32)
    W.set_lse_rows(w, full)
    want_out = oracle.softmax_l1_norm_rows(w.q_bits, w.k_bits, w.softmax_lse, sel, **kw)
    got = out.cpu().numpy().reshape(w.n_tokens, -1)
    assert_close(got[sel], want_out, what=f"{w.name} fused out")
    has = ~np.isneginf(want_lse[:, 0])
    sums = got[sel].astype(np.float64).sum(axis=1)
    assert np.all(np.abs(sums[has] - 1.0) <= ROWSUM_TOL), f"row sums {sums[has].min()}..{sums[has].max()}"
    assert np.all(sums[~has] == 0.0)
    assert np.all(np.isfinite(got)) and np.all(got >= 0)
    return lse_rows, got


@pytest.mark.parametrize("G", [1, 8, 64, 100, 128])
def test_lse_sparse_heads_multi_tile_ragged(lib, G):
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=24, S2=700, G=G, topk=300, mask_mode=3,
                        seed=5000 + G, lse=None)
    lse_parity(lib, w)


@pytest.mark.parametrize("G", [1, 5, 16, 128])
def test_lse_dense_heads_causal(lib, G):
    """Dense form: R = 128 // G tokens per item, each row with its own causal limit."""
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=37, S2=300, G=G, topk=0, mask_mode=3,
                        seed=5100 + G, lse=None)
    lse_parity(lib, w)


def test_lse_dense_no_mask(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=20, S2=257, G=8, topk=0, mask_mode=0,
                        seed=5200, lse=None)
    lse_parity(lib, w)


def test_lse_tnd_sparse_varlen_with_empty_sequences(lib):
    w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[130, 1, 0, 77, 260],
                        seqlens_k=[130, 5, 3, 200, 260], G=64, topk=256, mask_mode=3, seed=5300, lse=None)
    lse_parity(lib, w)


def test_lse_tnd_dense_width_beyond_sequences(lib):
    w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[40, 9, 70], seqlens_k=[50, 9, 130], G=16,
                        topk=0, mask_mode=3, max_seqlen_k=150, seed=5400, lse=None)
    lse_parity(lib, w)


def test_lse_rows_without_keys_are_neg_inf(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=40, S2=16, G=8, topk=0, mask_mode=3,
                        seed=5500, lse=None)
    lse, got = lse_parity(lib, w)
    assert np.all(np.isneginf(lse[:24])) and np.all(got[:24] == 0.0)


def test_lse_bad_indices_masked_and_reported(lib):
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=6, S2=300, G=16, topk=200, mask_mode=3,
                        seed=5600, lse=None, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(5600))
    w.sparse_indices = rng.integers(-3, 330, size=w.sparse_indices.shape).astype(np.int32)
    lse_parity(lib, w, expect=lib.SMLA_WARN_BAD_INDEX)


def test_lse_topk_length_cuts_real_keys(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=8, S2=512, G=32, topk=256, mask_mode=0,
                        seed=5700, lse=None)
    w.topk_length.reshape(-1)[:] = [0, -5, 1, 255, 256, 999, 128, 129]
    lse, _ = lse_parity(lib, w)
    assert np.all(np.isneginf(lse[:2]))


def test_lse_seqused(lib):
    w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[70, 9, 130], seqlens_k=[90, 9, 200], G=16,
                        topk=0, mask_mode=3, max_seqlen_k=220, seed=5800, lse=None)
    lse_parity(lib, w, su_q=[50, 9, 3], su_k=[1000, 0, 77])
    w = W.make_workload(layout="BSND", dtype="bf16", B=3, S1=40, S2=600, G=128, topk=300, mask_mode=3,
                        seed=5801, lse=None)
    lse_parity(lib, w, su_q=[40, 17, 0], su_k=[600, 250, 5])


def test_lse_large_logits_need_the_running_max(lib):
    """q and k entries in {-1, 0, 1} (exact in bf16, so every q.k is an
    exact integer in the fp32 accumulator) and softmax_scale 2.5: logits
    reach ~125, beyond fp32 exp's range, so the LSE only comes out finite
    with the running maximum."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=6, S2=600, G=16, topk=512, mask_mode=3,
                        seed=5900, lse=None, scale=2.5)
    rng = np.random.Generator(np.random.PCG64(5900))
    w.q_bits = W.bf16_bits_from_f32(rng.integers(-1, 2, size=w.q_bits.shape).astype(np.float32))
    w.k_bits = W.bf16_bits_from_f32(rng.integers(-1, 2, size=w.k_bits.shape).astype(np.float32))
    lse, _ = lse_parity(lib, w)
    assert lse.max() > 89.0


@pytest.mark.parametrize("n", [3, 4, 5])
def test_lse_full_size_sampled(lib, n):
    """Full-size configuration in the launch configuration the benchmark
    times; the oracle checks a sample of rows."""
    w = W.make_config(n)
    rng = np.random.Generator(np.random.PCG64(77 + n))
    rows = sorted(set([0, 1, w.n_tokens - 1, w.n_tokens // 2] +
                      rng.choice(w.n_tokens, 20, replace=False).tolist()))
    lse_parity(lib, w, rows=rows)
