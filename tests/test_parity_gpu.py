"""GPU parity: the CUDA library against the fp64 oracle, element by element,
through the C ABI.  Tolerance |gpu - oracle| <= 1e-5 + 2e-3 |oracle|; row sums
within 1e-3 of 1 where the LSE is the exact forward LSE."""
import numpy as np
import pytest

import oracle
import workloads as W
from smla_harness import (ROWSUM_TOL, assert_close, exact_lse, invalid_slot_mask, oracle_kwargs,
                          plan_kwargs, run_gpu, to_device)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def full_parity(smla, w, check_rowsum=True, **plan_extra):
    exact_lse(oracle, w)
    got, plan, t, status = run_gpu(smla, w, **plan_extra)
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    assert got.shape == want.shape
    assert_close(got, want, what=w.name)
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    bad = invalid_slot_mask(w)
    assert np.all(rows[bad] == 0.0), "masked / padding slots must be exactly 0"
    if check_rowsum:
        lse = w.lse_rows()
        has = ~np.isneginf(lse[:, 0])
        sums = rows.sum(axis=1)
        assert np.all(np.abs(sums[has] - 1.0) <= ROWSUM_TOL), f"row sums {sums[has].min()}..{sums[has].max()}"
        assert np.all(sums[~has] == 0.0)
    return got, plan, status


def test_config1_tiny_sparse(lib):
    w = W.make_config(1, lse=None)
    _, plan, status = full_parity(lib, w)
    assert status[0] == lib.SMLA_OK


def test_config2_dense_causal(lib):
    w = W.make_config(2, lse=None)
    _, plan, status = full_parity(lib, w)
    assert plan.info.rows_per_item == 8 and status[0] == lib.SMLA_OK


@pytest.mark.parametrize("G", [1, 3, 8, 16, 24, 64, 100, 128])
def test_sparse_head_counts_multi_tile_ragged(lib, G):
    """Several 128-key tiles plus a ragged tail (topk 300), causal, bf16."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=24, S2=700, G=G, topk=300,
                        mask_mode=3, seed=1000 + G, lse=None)
    full_parity(lib, w)


@pytest.mark.parametrize("G", [1, 5, 16, 48, 128])
def test_dense_head_counts(lib, G):
    """Dense form: R = 128 // G tokens packed per MMA, causal with S1 < S2."""
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=37, S2=300, G=G, topk=0,
                        mask_mode=3, seed=2000 + G, lse=None)
    full_parity(lib, w)


def test_dense_no_mask_bf16(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=20, S2=257, G=8, topk=0,
                        mask_mode=0, seed=2100, lse=None)
    full_parity(lib, w)


def test_tnd_sparse_varlen(lib):
    w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[130, 1, 0, 77, 260],
                        seqlens_k=[130, 5, 3, 200, 260], G=64, topk=256, mask_mode=3,
                        seed=2200, lse=None)
    full_parity(lib, w)


def test_tnd_dense_width_beyond_sequences(lib):
    w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[40, 9, 70],
                        seqlens_k=[50, 9, 130], G=16, topk=0, mask_mode=3, max_seqlen_k=150,
                        seed=2300, lse=None)
    full_parity(lib, w)


def test_s1_longer_than_s2_rows_without_keys(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=40, S2=16, G=8, topk=0,
                        mask_mode=3, seed=2400, lse=None)
    got, _, _ = full_parity(lib, w)
    assert np.all(got.reshape(40, -1)[:24] == 0.0)


def test_no_key_rows_at_all(lib):
    """S2 = 0: no key row exists, every slot is masked; the output is all
    zero and the forward LSE is -inf (k may be NULL).  No key tile runs."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=5, S2=0, G=16, topk=8, mask_mode=0,
                        seed=2450, lse=None, with_topk_length=False)
    w.sparse_indices = np.full(w.sparse_indices.shape, -1, np.int32)
    W.set_lse_rows(w, np.zeros((w.n_tokens, w.G), np.float32))
    plan = lib.Plan(**plan_kwargs(w))
    t = to_device(w)
    out = plan.run(t["q"], None, t["lse"], sparse_indices=t["idx"])
    lse = plan.softmax_lse(t["q"], None, sparse_indices=t["idx"])
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == 0.0)
    assert np.all(np.isneginf(lse.cpu().numpy()))
    assert plan.status()[0] == lib.SMLA_OK  # no tile runs, so no index is read


@pytest.mark.parametrize("topk,S2", [(8192, 9000), (1001, 1500)])
def test_large_and_ragged_topk(lib, topk, S2):
    """64 key tiles per token, and a topk that is no multiple of 4 or 16."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=6, S2=S2, G=16, topk=topk, mask_mode=0,
                        seed=2460 + topk, lse=None)
    full_parity(lib, w)


def test_bad_indices_are_masked_and_reported(lib):
    """No topk_length: every slot is a candidate; -1 is padding, other values
    outside [0, Sk) are masked and raise the bad-index warning."""
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=6, S2=300, G=16, topk=200,
                        mask_mode=3, seed=2500, lse=None, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(2500))
    w.sparse_indices = rng.integers(-3, 330, size=w.sparse_indices.shape).astype(np.int32)
    _, _, status = full_parity(lib, w)
    assert status[0] == lib.SMLA_WARN_BAD_INDEX and (status[1] & 1)


def test_topk_length_clamped_and_zero(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=8, S2=512, G=32, topk=256,
                        mask_mode=0, seed=2600, lse=None)
    tl = w.topk_length.reshape(-1)
    tl[:] = [0, -5, 1, 255, 256, 999, 128, 129]
    # the oracle reads topk_length as "slot < topk_length"; clamping to [0, topk] is the same
    full_parity(lib, w)


def test_empty_q_returns_at_once(lib):
    plan = lib.Plan(layout="BSND", dtype="bf16", num_heads_q=8, batch_size=0, max_seqlen_q=16,
                    max_seqlen_k=64, topk=8, mask_mode=0, softmax_scale=1.0)
    assert plan.output_shape == (0, 16, 1, 8)
    code = plan._lib.smla_l1norm_run(plan._h, None, None, None, None, None, None, None)
    assert code == lib.SMLA_OK


def test_deterministic_bitwise(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=200, S2=2048, G=128, topk=1024,
                        mask_mode=3, seed=2700)
    a, plan, t, _ = run_gpu(lib, w)
    b, _, _, _ = run_gpu(lib, w, plan=plan, tensors=t)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # another grid size gives the same bits (the schedule only moves work)
    c, _, _, _ = run_gpu(lib, w, tensors=t, num_ctas=7)
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32))


def test_run_from_host_matches_run(lib):
    w = W.make_config(1)
    a, plan, t, _ = run_gpu(lib, w)
    pin = {k: (None if v is None else v.cpu().pin_memory()) for k, v in
           {"q": t["q"], "k": t["k"], "lse": t["lse"], "indices": t["idx"], "topk_length": t["tl"]}.items()}
    pin["out"] = torch.empty(plan.output_shape, dtype=torch.float32).pin_memory()
    dev = {"q": torch.empty_like(t["q"]), "k": torch.empty_like(t["k"]), "lse": torch.empty_like(t["lse"]),
           "indices": torch.empty_like(t["idx"]), "topk_length": torch.empty_like(t["tl"]),
           "out": torch.empty(plan.output_shape, dtype=torch.float32, device="cuda")}
    plan.run_from_host(pin, dev)
    torch.cuda.synchronize()
    assert np.array_equal(pin["out"].numpy(), a)


@pytest.mark.parametrize("kind", ["sparse_bsnd", "dense_tnd"])
def test_run_from_host_pipelined_matches_run(lib, kind):
    """With 8 CTAs every workload below has enough items for the token-chunk
    pipeline of run_from_host; its output equals run()'s bit for bit."""
    if kind == "sparse_bsnd":
        w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=100, S2=900, G=32, topk=512,
                            mask_mode=3, seed=2850)
    else:
        w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[70, 130, 40], seqlens_k=[90, 130, 60],
                            G=64, topk=0, mask_mode=3, seed=2851)
    a, plan, t, _ = run_gpu(lib, w, num_ctas=8)
    assert plan.info.host_chunks >= 4
    pin = {k: (None if v is None else v.cpu().pin_memory()) for k, v in
           {"q": t["q"], "k": t["k"], "lse": t["lse"], "indices": t["idx"], "topk_length": t["tl"]}.items()}
    pin["out"] = torch.full(plan.output_shape, float("nan"), dtype=torch.float32).pin_memory()
    dev = {"q": torch.empty_like(t["q"]), "k": torch.empty_like(t["k"]), "lse": torch.empty_like(t["lse"]),
           "indices": None if t["idx"] is None else torch.empty_like(t["idx"]),
           "topk_length": None if t["tl"] is None else torch.empty_like(t["tl"]),
           "out": torch.empty(plan.output_shape, dtype=torch.float32, device="cuda")}
    for _ in range(2):  # twice: the second call reuses the plan's streams and events
        plan.run_from_host(pin, dev)
        torch.cuda.synchronize()
        assert np.array_equal(pin["out"].numpy().view(np.uint32), a.view(np.uint32))
        pin["out"].fill_(float("nan"))


def test_run_is_capturable_in_a_cuda_graph(lib):
    """run() does host work only to encode the q tensor map and launches one
    kernel (no allocation, no synchronisation), so it can be captured in a
    CUDA graph; replays give the eager result bit for bit."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=64, S2=1000, G=128, topk=512, mask_mode=3,
                        seed=2860)
    a, plan, t, _ = run_gpu(lib, w)
    out = torch.full(plan.output_shape, float("nan"), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"], out=out, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"], out=out)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), a.view(np.uint32))
    assert plan.status()[0] == lib.SMLA_OK


def test_functional_api_matches_plan(lib):
    w = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[33, 70], seqlens_k=[33, 90], G=16,
                        topk=64, mask_mode=3, seed=2800)
    a, _, t, _ = run_gpu(lib, w)
    b = lib.sparse_flash_mla_softmax_l1_norm(
        t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"],
        cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k, softmax_scale=w.softmax_scale,
        mask_mode=3, layout_q="TND", layout_k="TND")
    assert np.array_equal(b.cpu().numpy(), a)


def test_wait_timeout_probe_reports_and_returns(lib):
    code, flags = lib.wait_timeout_probe(50_000_000)
    assert code == lib.SMLA_ERR_TIMEOUT and (flags & 2)
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0


@pytest.mark.parametrize("topk,S2,mask", [(300, 700, 3), (128, 400, 0), (2048, 2100, 3)])
def test_cta_pair_kernel(lib, monkeypatch, topk, S2, mask):
    """Sparse form with 128 heads: the L1-norm launch runs on 2-CTA clusters
    (one MMA over both CTAs' keys; forced here, chosen by the plan for long
    tokens).  Odd and even tile counts per token,
    tokens whose causal limit cuts the tiles; compared with the oracle
    element by element and with the single-CTA kernel (SMLA_PAIR=0)."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=40, S2=S2, G=128, topk=topk, mask_mode=mask,
                        seed=7000 + topk, lse=None)
    exact_lse(oracle, w)
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    t = to_device(w)
    monkeypatch.setenv("SMLA_PAIR", "1")   # forced: the plan picks one CTA for the short tokens
    got, plan, _, status = run_gpu(lib, w, tensors=t)
    assert plan.info.cta_pairs > 0 and status[0] == lib.SMLA_OK
    assert_close(got, want, what="CTA pair kernel")
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    assert np.all(rows[invalid_slot_mask(w)] == 0.0)
    assert np.all(np.abs(rows.sum(axis=1) - 1.0) <= ROWSUM_TOL)
    monkeypatch.setenv("SMLA_PAIR", "0")
    single, plan1, _, _ = run_gpu(lib, w, tensors=t)
    assert plan1.info.cta_pairs == 0
    assert_close(single, want, what="single-CTA kernel")
    again, _, _, _ = run_gpu(lib, w, plan=plan, tensors=t)
    assert np.array_equal(again.view(np.uint32), got.view(np.uint32)), "pair kernel run to run"
    # a grid size the caller asks for bounds the pairs too; the bits do not change
    monkeypatch.setenv("SMLA_PAIR", "1")
    small, plan7, _, _ = run_gpu(lib, w, tensors=t, num_ctas=7)
    assert plan7.info.cta_pairs == 3
    assert np.array_equal(small.view(np.uint32), got.view(np.uint32)), "pair kernel on 3 clusters"
    # one CTA asked for: no pair, and the single-CTA kernel's bits on one SM
    one, plan1c, _, _ = run_gpu(lib, w, tensors=t, num_ctas=1)
    assert plan1c.info.cta_pairs == 0 and plan1c.info.num_ctas == 1
    assert np.array_equal(one.view(np.uint32), single.view(np.uint32)), "single-CTA kernel on one CTA"


def test_fused_kernel_waits_give_up_and_report(lib, monkeypatch):
    """A plan whose launches never load one q chunk (a test hook) and whose
    device waits are bounded by 30 ms: the MMA issuers' wait for that chunk
    runs out, sets the CTA's abort flag and the timeout bit; every role leaves
    its loop, copies and MMAs in flight are drained and TMEM is released.
    Each launch mode reports SMLA_ERR_TIMEOUT -- the L1-norm launch on the
    single-CTA kernel and on the CTA-pair kernel (forced) -- and afterwards
    the context still computes the oracle's result with a normal plan."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=64, S2=2500, G=128, topk=2048, mask_mode=3,
                        seed=5200, lse=None)
    exact_lse(oracle, w)
    t = to_device(w)
    monkeypatch.setenv("SMLA_WAIT_TIMEOUT_MS", "30")
    monkeypatch.setenv("SMLA_DEBUG_WITHHOLD_Q", "1")
    monkeypatch.setenv("SMLA_PAIR", "0")
    plan0 = lib.Plan(**plan_kwargs(w))
    monkeypatch.setenv("SMLA_PAIR", "1")
    plan_pair = lib.Plan(**plan_kwargs(w))
    monkeypatch.delenv("SMLA_PAIR")
    monkeypatch.delenv("SMLA_WAIT_TIMEOUT_MS")
    monkeypatch.delenv("SMLA_DEBUG_WITHHOLD_Q")
    assert plan0.info.cta_pairs == 0 and plan_pair.info.cta_pairs > 0
    runs = {
        "l1": (plan0, lambda: plan0.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"])),
        "l1 pair": (plan_pair, lambda: plan_pair.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"],
                                                     topk_length=t["tl"])),
        "lse": (plan0, lambda: plan0.softmax_lse(t["q"], t["k"], sparse_indices=t["idx"], topk_length=t["tl"])),
        "fused": (plan0, lambda: plan0.run_fused_lse(t["q"], t["k"], sparse_indices=t["idx"], topk_length=t["tl"])),
    }
    for name, (pl, fn) in runs.items():
        fn()
        torch.cuda.synchronize()
        code, flags = pl.status()
        assert code == lib.SMLA_ERR_TIMEOUT and (flags & 2), (name, code, flags)
    got, plan, _, status = run_gpu(lib, w, tensors=t)
    assert status[0] == lib.SMLA_OK
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    assert_close(got, want, what="normal plan after the aborted launches")


# ---------------------------------------------------------------- full sizes
def rows_from_every_cta(lib, w, plan, rng):
    """One query token from each CTA's item list of ``plan``'s schedule (the
    host scheduler builds the same list for the same description and grid)."""
    items, offs, _ = lib.schedule_host(plan.info.num_ctas, **plan_kwargs(w))
    rows = []
    for c in range(len(offs) - 1):
        if offs[c + 1] > offs[c]:
            it = items[int(rng.integers(offs[c], offs[c + 1]))]
            rows.append(int(it[0]) + int(rng.integers(0, it[1])))
    return rows


def sampled_parity(lib, n, n_sample=24, seed=0):
    """Full-size configuration, in the launch configuration the benchmark
    times.  Exact LSE is planted for a sample of rows -- one from every CTA's
    share of the schedule plus random ones -- which are compared element by
    element with the oracle and must sum to 1; every row is checked for exact
    zeros on invalid slots and for finite, non-negative values."""
    w = W.make_config(n)
    rng = np.random.Generator(np.random.PCG64(seed))
    n_tok = w.n_tokens
    plan = lib.Plan(**plan_kwargs(w))
    rows = set([0, 1, n_tok - 1, n_tok // 2] + rng.choice(n_tok, n_sample, replace=False).tolist())
    per_cta = rows_from_every_cta(lib, w, plan, rng)
    assert len(per_cta) == plan.info.num_ctas
    rows = sorted(rows | set(per_cta))
    exact_lse(oracle, w, rows=rows)
    got, plan, t, status = run_gpu(lib, w, plan=plan)
    assert status[0] == lib.SMLA_OK
    got_rows = got.reshape(n_tok, -1)
    want = oracle.softmax_l1_norm_rows(w.q_bits, w.k_bits, w.softmax_lse, rows, **oracle_kwargs(w))
    assert_close(got_rows[rows], want, what=f"config {n} sampled rows")
    sums = got_rows[rows].astype(np.float64).sum(axis=1)
    assert np.all(np.abs(sums - 1.0) <= ROWSUM_TOL), sums
    assert np.all(np.isfinite(got_rows)) and np.all(got_rows >= 0)
    bad = invalid_slot_mask(w)
    assert np.all(got_rows[bad] == 0.0)
    return w, got_rows


def test_config3_dsv32_full_size_every_row(lib, tmp_path, monkeypatch):
    """The 4096-token, 128-head, top-2048 causal workload at full size, in the
    benchmark's launch configuration: the exact forward LSE is planted on
    every row and every one of the 8.4 M output elements is compared with the
    oracle; every row sums to 1 within 1e-3 and masked slots are exactly 0.
    The plan picks the CTA-pair kernel for this workload (12.3 key tiles a
    token); then the same with the single-CTA kernel forced."""
    import oracle_pool
    w = W.make_config(3)
    n_tok = w.n_tokens
    lse, want = oracle_pool.lse_and_rows(w, range(n_tok), str(tmp_path / "c3"))
    W.set_lse_rows(w, lse)
    monkeypatch.delenv("SMLA_PAIR", raising=False)
    got_pair, plan_pair, t, status = run_gpu(lib, w)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert status[0] == lib.SMLA_OK and plan_pair.info.cta_pairs > 0
    monkeypatch.setenv("SMLA_PAIR", "0")
    got, plan, _, status = run_gpu(lib, w, tensors=t)
    assert status[0] == lib.SMLA_OK and plan.info.cta_pairs == 0 and plan.info.num_ctas == n_sm
    for name, g in (("CTA-pair", got_pair), ("single-CTA", got)):
        got_rows = g.reshape(n_tok, -1)
        assert_close(got_rows, want, what=f"config 3, every element, {name} kernel")
        sums = got_rows.astype(np.float64).sum(axis=1)
        assert np.all(np.abs(sums - 1.0) <= ROWSUM_TOL), (name, sums.min(), sums.max())
        assert np.all(got_rows[invalid_slot_mask(w)] == 0.0)


def test_config4_varlen_tnd_full_size_sampled(lib):
    sampled_parity(lib, 4)


def test_config5_long_clustered_full_size_sampled(lib):
    sampled_parity(lib, 5, n_sample=16)


# ---------------------------------------------------------------- seqused_q / seqused_k
def seqused_parity(lib, w, su_q, su_k):
    """Parity with per-sequence participating lengths.  The LSE is the exact
    forward LSE over the cut problem, so every row with a kept slot sums to
    1; rows past seqused_q and slots past seqused_k are exactly 0."""
    kw = oracle_kwargs(w)
    kw.update(seqused_q=su_q, seqused_k=su_k)
    W.set_lse_rows(w, oracle.softmax_lse(w.q_bits, w.k_bits, **kw).astype(np.float32))
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw)
    plan = lib.Plan(**plan_kwargs(w))
    t = to_device(w)
    dev = lambda v: None if v is None else torch.tensor(np.asarray(v, np.int32), device="cuda")
    out = plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"],
                   seqused_q=dev(su_q), seqused_k=dev(su_k))
    torch.cuda.synchronize()
    code, _ = plan.status()
    assert code == lib.SMLA_OK
    got = out.cpu().numpy()
    assert_close(got, want, what=w.name)
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    assert np.all(rows[want.reshape(w.n_tokens, -1) == 0.0] == 0.0), "cut slots must be exactly 0"
    has = ~np.isneginf(w.lse_rows()[:, 0])
    assert np.all(np.abs(rows[has].sum(axis=1) - 1.0) <= ROWSUM_TOL)
    assert np.all(rows[~has] == 0.0)
    return got


def test_seqused_sparse_bsnd(lib):
    w = W.make_workload(name="seqused_sparse", layout="BSND", dtype="bf16", B=3, S1=40, S2=600, G=16,
                        topk=300, mask_mode=3, seed=3100, lse=None)
    got = seqused_parity(lib, w, su_q=[40, 17, 0], su_k=[600, 250, 5])
    g = got.reshape(3, 40, -1)
    assert np.all(g[1, 17:] == 0.0) and np.all(g[2] == 0.0)


def test_seqused_sparse_tnd_keys_only_and_negative(lib):
    w = W.make_workload(name="seqused_sparse_tnd", layout="TND", dtype="fp16", seqlens_q=[130, 1, 77],
                        seqlens_k=[130, 5, 300], G=64, topk=256, mask_mode=0, seed=3101, lse=None)
    seqused_parity(lib, w, su_q=None, su_k=[-4, 9, 129])


def test_seqused_dense_tnd(lib):
    w = W.make_workload(name="seqused_dense_tnd", layout="TND", dtype="bf16", seqlens_q=[70, 9, 130],
                        seqlens_k=[90, 9, 200], G=16, topk=0, mask_mode=3, max_seqlen_k=220,
                        seed=3102, lse=None)
    seqused_parity(lib, w, su_q=[50, 9, 3], su_k=[1000, 0, 77])


def test_seqused_dense_shorter_queries_see_more_keys(lib):
    """Cutting Sq moves the right-down causal diagonal: with Sq' = 20 and
    Sk = 64, row 0 sees keys 0..44."""
    w = W.make_workload(name="seqused_diag", layout="BSND", dtype="fp16", B=1, S1=64, S2=64, G=8,
                        topk=0, mask_mode=3, seed=3103, lse=None)
    got = seqused_parity(lib, w, su_q=[20], su_k=None).reshape(64, 64)
    nz = (got != 0.0).sum(axis=1)
    assert nz[0] == 45 and nz[19] == 64 and np.all(nz[20:] == 0)


def test_seqused_full_lengths_bitwise_equal_to_run(lib):
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=33, S2=700, G=128, topk=512,
                        mask_mode=3, seed=3104)
    a, plan, t, _ = run_gpu(lib, w)
    full = torch.tensor([33, 33], dtype=torch.int32, device="cuda")
    fullk = torch.tensor([700, 700], dtype=torch.int32, device="cuda")
    b = plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], topk_length=t["tl"],
                 seqused_q=full, seqused_k=fullk)
    torch.cuda.synchronize()
    assert np.array_equal(a.view(np.uint32), b.cpu().numpy().view(np.uint32))


# ---------------------------------------------------------------- dense key split
@pytest.mark.parametrize("split", [1, 2, 4])
@pytest.mark.parametrize("mask", [0, 3])
def test_dense_split_along_keys(lib, monkeypatch, split, mask):
    """Dense L1-norm launch with each token pack's key tiles split into parts
    (forced with SMLA_SPLIT; the plan splits by itself only when few long
    packs would unbalance the grid).  6 key tiles and a ragged tail per
    pack; parts zero only their own uncomputed range, the last part the rest
    of the row.  Compared with the oracle, and bit for bit with the unsplit
    launch: a slot's sum over the heads is computed the same way by
    whichever CTA owns it."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=50, S2=700, G=16, topk=0, mask_mode=mask,
                        seed=7300 + split + 10 * mask, lse=None)
    exact_lse(oracle, w)
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    t = to_device(w)
    monkeypatch.setenv("SMLA_SPLIT", str(split))
    got, plan, _, status = run_gpu(lib, w, tensors=t)
    assert plan.info.split_tiles == split and plan.info.split_items > plan.info.num_items
    assert status[0] == lib.SMLA_OK
    assert_close(got, want, what=f"dense split {split}")
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    assert np.all(rows[invalid_slot_mask(w)] == 0.0)
    assert np.all(np.abs(rows.sum(axis=1) - 1.0) <= ROWSUM_TOL)
    monkeypatch.setenv("SMLA_SPLIT", "0")
    whole, plan0, _, _ = run_gpu(lib, w, tensors=t)
    assert plan0.info.split_tiles == 0
    assert np.array_equal(whole.view(np.uint32), got.view(np.uint32))
    # the forward LSE launch of a split plan takes whole packs
    lse = plan.softmax_lse(t["q"], t["k"])
    torch.cuda.synchronize()
    l = lse.cpu().numpy().reshape(w.n_tokens, w.G).astype(np.float64)
    ref = w.lse_rows().astype(np.float64)
    assert np.all(np.abs(l - ref) <= 1e-4 + 1e-6 * np.abs(ref))


def test_dense_split_with_seqused_and_compressed_keys(lib, monkeypatch):
    """Parts of a split pack under seqused_q / seqused_k (the pack's visible
    tiles end inside or before a part) and with compressed keys."""
    monkeypatch.setenv("SMLA_SPLIT", "1")
    w = W.make_workload(name="split_seqused", layout="TND", dtype="bf16", seqlens_q=[70, 9, 130],
                        seqlens_k=[400, 9, 300], G=16, topk=0, mask_mode=3, max_seqlen_k=420,
                        seed=7310, lse=None)
    seqused_parity(lib, w, su_q=[50, 9, 3], su_k=[1000, 0, 200])
    w = W.make_workload(name="split_cmp", layout="BSND", dtype="fp16", B=2, S1=300, S2=400, G=16, topk=0,
                        mask_mode=3, seed=7311, lse=None)
    res = np.asarray([1, 3], np.int32)
    okw = dict(oracle_kwargs(w), cmp_ratio=4, cmp_residual_k=res)
    W.set_lse_rows(w, oracle.softmax_lse(w.q_bits, w.k_bits, **okw).astype(np.float32))
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **okw)
    plan = lib.Plan(**plan_kwargs(w, cmp_ratio=4))
    assert plan.info.split_tiles == 1
    t = to_device(w)
    out = plan.run(t["q"], t["k"], t["lse"], cmp_residual_k=torch.tensor(res, device="cuda"))
    torch.cuda.synchronize()
    assert plan.status()[0] == lib.SMLA_OK
    assert_close(out.cpu().numpy(), want, what="split, compressed keys")


def test_config2_plan_splits_by_itself(lib):
    """The 2 x 512 causal dense workload (128 packs of 1-4 key tiles for 152
    CTAs) is split by the plan without any override; full parity is the
    config-2 test above."""
    w = W.make_config(2)
    plan = lib.Plan(**plan_kwargs(w))
    assert plan.info.split_tiles > 0 and plan.info.split_items > plan.info.num_items


# ---------------------------------------------------------------- CTA pairs under cut lengths / compressed keys
def test_cta_pair_kernel_with_seqused(lib, monkeypatch):
    """The CTA-pair kernel (forced) under seqused_q / seqused_k: rows past
    seqused_q are zero, keys past seqused_k masked, the causal diagonal on
    the cut lengths; against the oracle, and against the single-CTA kernel
    (within the tolerance: the two kernels split the head dimension
    between their issuers differently, so fp32 partial sums round apart)."""
    monkeypatch.setenv("SMLA_PAIR", "1")
    w = W.make_workload(name="pair_seqused", layout="BSND", dtype="bf16", B=3, S1=30, S2=1500, G=128,
                        topk=1100, mask_mode=3, seed=7400, lse=None)
    got = seqused_parity(lib, w, su_q=[30, 11, 0], su_k=[1500, 700, 9])
    monkeypatch.setenv("SMLA_PAIR", "0")
    single = seqused_parity(lib, w, su_q=[30, 11, 0], su_k=[1500, 700, 9])
    assert_close(got, single, what="pair vs single-CTA kernel")
    assert np.array_equal(got == 0.0, single == 0.0)


def test_cta_pair_kernel_with_compressed_keys(lib, monkeypatch):
    """The CTA-pair kernel (forced) with compressed keys of ratio 4 and
    per-sequence residuals under the causal mask."""
    monkeypatch.setenv("SMLA_PAIR", "1")
    w = W.make_workload(name="pair_cmp", layout="BSND", dtype="bf16", B=2, S1=64, S2=600, G=128, topk=700,
                        mask_mode=3, seed=7401, lse=None, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(7401))
    w.sparse_indices = rng.integers(-1, 620, size=w.sparse_indices.shape).astype(np.int32)
    res = np.asarray([0, 3], np.int32)
    okw = dict(oracle_kwargs(w), cmp_ratio=4, cmp_residual_k=res)
    W.set_lse_rows(w, oracle.softmax_lse(w.q_bits, w.k_bits, **okw).astype(np.float32))
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **okw)
    plan = lib.Plan(**plan_kwargs(w, cmp_ratio=4))
    assert plan.info.cta_pairs > 0
    t = to_device(w)
    out = plan.run(t["q"], t["k"], t["lse"], sparse_indices=t["idx"], cmp_residual_k=torch.tensor(res, device="cuda"))
    torch.cuda.synchronize()
    assert plan.status()[0] in (lib.SMLA_OK, lib.SMLA_WARN_BAD_INDEX)
    got = out.cpu().numpy()
    assert_close(got, want, what="CTA pairs, compressed keys")
    rows = got.reshape(w.n_tokens, -1).astype(np.float64)
    assert np.all(rows[want.reshape(w.n_tokens, -1) == 0.0] == 0.0)
    has = ~np.isneginf(w.lse_rows()[:, 0])
    assert np.all(np.abs(rows[has].sum(axis=1) - 1.0) <= ROWSUM_TOL)


def pair_and_single(lib, monkeypatch, w):
    """Oracle parity of the CTA-pair kernel (forced) and of the single-CTA
    kernel (forced) on the same inputs; returns both outputs and statuses."""
    exact_lse(oracle, w)
    want = oracle.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **oracle_kwargs(w))
    t = to_device(w)
    bad = invalid_slot_mask(w)
    has = ~np.isneginf(w.lse_rows()[:, 0])
    res = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("SMLA_PAIR", mode)
        got, plan, _, status = run_gpu(lib, w, tensors=t)
        assert (plan.info.cta_pairs > 0) == (mode == "1")
        name = "CTA-pair" if mode == "1" else "single-CTA"
        assert_close(got, want, what=f"{w.name}, {name} kernel")
        rows = got.reshape(w.n_tokens, -1).astype(np.float64)
        assert np.all(rows[bad] == 0.0), name
        assert np.all(np.abs(rows[has].sum(axis=1) - 1.0) <= ROWSUM_TOL), name
        res[mode] = (got, status)
    return res


def test_cta_pair_kernel_tnd_varlen(lib, monkeypatch):
    """TND layout with 128 heads, queries shorter than their keys (the
    right-down causal diagonal lets early queries see long prefixes), one
    sequence with a single query and one with none: the CTA-pair kernel
    against the oracle and against the single-CTA kernel."""
    w = W.make_workload(name="pair_tnd", layout="TND", dtype="fp16", seqlens_q=[300, 1, 0, 260, 90],
                        seqlens_k=[1500, 5, 3, 2100, 1300], G=128, topk=1536, mask_mode=3, seed=7402, lse=None)
    res = pair_and_single(lib, monkeypatch, w)
    assert res["1"][1][0] == lib.SMLA_OK and res["0"][1][0] == lib.SMLA_OK
    assert np.array_equal(res["1"][0] == 0.0, res["0"][0] == 0.0)


def test_cta_pair_kernel_without_topk_length_bad_indices(lib, monkeypatch):
    """No topk_length: all 2048 slots are candidates, with -1 padding and
    out-of-range indices spread through them (masked and reported by both
    kernels)."""
    w = W.make_workload(name="pair_bad_idx", layout="BSND", dtype="bf16", B=2, S1=24, S2=2200, G=128, topk=2048,
                        mask_mode=3, seed=7403, lse=None, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(7403))
    w.sparse_indices = rng.integers(-3, 2300, size=w.sparse_indices.shape).astype(np.int32)
    res = pair_and_single(lib, monkeypatch, w)
    for mode in ("1", "0"):
        assert res[mode][1][0] == lib.SMLA_WARN_BAD_INDEX and (res[mode][1][1] & 1)


@pytest.mark.parametrize("G", [113, 120, 127])
def test_cta_pairs_only_for_exactly_128_heads(lib, monkeypatch, G):
    """Head counts of 113-127 pad the MMA's N to 128 as well, but the CTA-pair
    kernel splits q into two 64-head halves and reads 128 LSE entries a
    token: the plan keeps such work on one CTA per SM, even when pairs are
    forced, and the result matches the oracle."""
    w = W.make_workload(name=f"g{G}_long", layout="BSND", dtype="bf16", B=1, S1=12, S2=2100, G=G, topk=2048,
                        mask_mode=3, seed=7500 + G, lse=None)
    for mode in (None, "1"):
        if mode is None:
            monkeypatch.delenv("SMLA_PAIR", raising=False)
        else:
            monkeypatch.setenv("SMLA_PAIR", mode)
        got, plan, status = full_parity(lib, w)
        assert plan.info.cta_pairs == 0 and status[0] == lib.SMLA_OK
