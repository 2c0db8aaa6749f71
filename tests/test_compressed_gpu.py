"""Compressed keys on the GPU (cmp_ratio 2..128 with cmp_residual_k, article
"SparseFlashMlaSoftmaxL1Norm", parameter table 参数说明 and constraints
约束说明), through the C ABI, against the oracle element by element.

Reading: key j of K stands for original positions j*c .. j*c + c - 1 of an
original key sequence of Sk*c + cmp_residual_k positions; right-down causal
keeps a key when its whole block is visible.  The exact forward LSE under the
same rule is planted on every row, so rows with a kept key sum to 1."""
import numpy as np
import pytest

import oracle
import workloads as W
from smla_harness import ROWSUM_TOL, assert_close, oracle_kwargs, plan_kwargs, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _dev(v):
    return None if v is None else torch.tensor(np.asarray(v, np.int32), device="cuda")


def cmp_parity(lib, w, c, res, seqused_q=None, seqused_k=None, random_indices=None):
    if random_indices is not None:
        rng = np.random.Generator(np.random.PCG64(w.seed))
        w.sparse_indices = rng.integers(random_indices[0], random_indices[1],
                                        size=w.sparse_indices.shape).astype(np.int32)
    res = None if res is None else np.asarray(res, np.int32)
    okw = dict(oracle_kwargs(w), cmp_ratio=c, cmp_residual_k=res, seqused_q=seqused_q, seqused_k=seqused_k)
    W.set_lse_rows(w, oracle.softmax_lse(w.q_bits, w.k_bits, **okw).astype(np.float32))
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **okw)
    plan = lib.Plan(**plan_kwargs(w, cmp_ratio=c))
    t = to_device(w)
    out = plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"],
                   seqused_q=_dev(seqused_q), seqused_k=_dev(seqused_k), cmp_residual_k=_dev(res))
    torch.cuda.synchronize()
    assert plan.status()[0] in (lib.SMLA_OK, lib.SMLA_WARN_BAD_INDEX)
    got = out.cpu().numpy()
    assert_close(got, want, what=f"{w.name} c={c}")
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    assert np.all(rows[want.reshape(w.n_tokens, -1) == 0.0] == 0.0), "masked slots must be exactly 0"
    has = ~np.isneginf(w.lse_rows()[:, 0])
    assert np.all(np.abs(rows[has].sum(axis=1) - 1.0) <= ROWSUM_TOL)
    assert np.all(rows[~has] == 0.0)
    return plan, t, got, okw


def test_compressed_sparse_bsnd_causal(lib):
    """100 queries over 30 compressed keys of ratio 4 (L = 120 + residual):
    row r keeps keys j < (r + 21 + res) // 4, so the residual moves the
    limit; indices include -1 and positions past the sequence."""
    w = W.make_workload(name="cmp_sparse", layout="BSND", dtype="bf16", B=2, S1=100, S2=30, G=16, topk=24,
                        mask_mode=3, seed=6100, lse=None, with_topk_length=False)
    plan, t, got, okw = cmp_parity(lib, w, 4, [0, 3], random_indices=(-1, 34))
    # the forward LSE and the fused launch under the same rule
    lse = plan.softmax_lse(t["q"], t["k"], sparse_indices=t["idx"], cmp_residual_k=_dev(okw["cmp_residual_k"]))
    out2, lse2 = plan.run_fused_lse(t["q"], t["k"], sparse_indices=t["idx"],
                                    cmp_residual_k=_dev(okw["cmp_residual_k"]))
    torch.cuda.synchronize()
    want_lse = w.lse_rows().astype(np.float64)
    for name, l in (("lse", lse), ("fused lse", lse2)):
        l = l.cpu().numpy().reshape(w.n_tokens, w.G).astype(np.float64)
        inf = np.isneginf(want_lse)
        assert np.array_equal(np.isneginf(l), inf), name
        assert np.all(np.abs(l[~inf] - want_lse[~inf]) <= 1e-4 + 1e-6 * np.abs(want_lse[~inf])), name
    assert_close(out2.cpu().numpy(), got, what="fused output")


def test_compressed_sparse_tnd_four_issuers(lib):
    """TND with per-sequence residuals, G = 64 (the four-issuer launch), c = 16."""
    w = W.make_workload(name="cmp_tnd", layout="TND", dtype="fp16", seqlens_q=[70, 5, 130],
                        seqlens_k=[9, 2, 20], G=64, topk=16, mask_mode=3, seed=6101, lse=None,
                        with_topk_length=False)
    plan, _, _, _ = cmp_parity(lib, w, 16, [15, 0, 7], random_indices=(-1, 21))
    assert plan.info.mma_issuers in (2, 4)


def test_compressed_dense_causal(lib):
    """Dense form, 8 tokens per MMA (G = 16), c = 8: a token's columns end at
    its own limit.  330 queries over L = 320 + res original positions: the
    first rows see no complete block and are all zero."""
    w = W.make_workload(name="cmp_dense", layout="BSND", dtype="bf16", B=2, S1=330, S2=40, G=16, topk=0,
                        mask_mode=3, seed=6102, lse=None)
    _, _, got, _ = cmp_parity(lib, w, 8, [2, 7])
    g = got.reshape(2, 330, 40)
    # row r keeps (r + 320 + res - 330 + 1) // 8 keys: the first kept key is
    # at row 15 (res 2) and row 10 (res 7)
    assert np.all(g[0, :15] == 0.0) and np.any(g[0, 15] != 0.0)
    assert np.all(g[1, :10] == 0.0) and np.any(g[1, 10] != 0.0)


def test_compressed_dense_tnd_with_seqused(lib):
    w = W.make_workload(name="cmp_dense_tnd", layout="TND", dtype="fp16", seqlens_q=[30, 12, 45],
                        seqlens_k=[20, 6, 33], G=8, topk=0, mask_mode=3, max_seqlen_k=40, seed=6103, lse=None)
    cmp_parity(lib, w, 4, [1, 3, 0], seqused_q=[30, 7, 40], seqused_k=[11, 6, 100])


def test_the_articles_tnd_call(lib):
    """The article's TND example: 16 queries (G = 128), 2048 compressed keys of
    ratio 128, residual 0, right-down causal, no sparse indices: output
    (16, 1, 2048); row r keeps (r + 2048*128 - 15) // 128 keys, i.e. 2047 for
    row 0 and all 2048 for row 15."""
    w = W.make_workload(name="article_tnd", layout="TND", dtype="fp16", seqlens_q=[16], seqlens_k=[2048],
                        G=128, topk=0, mask_mode=3, seed=6104, lse=None)
    plan, _, got, _ = cmp_parity(lib, w, 128, [0])
    assert got.shape == (16, 1, 2048) and plan.output_shape == (16, 1, 2048)
    kept = (got.reshape(16, 2048) != 0).sum(axis=1)
    assert list(kept) == [min(2048, (r + 2048 * 128 - 15) // 128) for r in range(16)]


def test_compressed_without_mask_equals_uncompressed(lib):
    """With mask 0 the ratio changes nothing: bit for bit the cmp_ratio = 1 output."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=20, S2=600, G=32, topk=300, mask_mode=0,
                        seed=6105)
    t = to_device(w)
    a = lib.Plan(**plan_kwargs(w)).run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"])
    b = lib.Plan(**plan_kwargs(w, cmp_ratio=64)).run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"],
                                                      topk_length=t["tl"])
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32))


def test_compressed_causal_needs_the_residual(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=8, S2=64, G=8, topk=16, mask_mode=3, seed=6106)
    plan = lib.Plan(**plan_kwargs(w, cmp_ratio=2))
    t = to_device(w)
    with pytest.raises(lib.SmlaError) as e:
        plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"])
    assert e.value.code == lib.SMLA_ERR_NULLPTR
