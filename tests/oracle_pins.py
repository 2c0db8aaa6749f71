"""Pins that tie the CPU oracle to what the definition fixes.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a library routine or a
brute-force loop.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with a planted
mistake and checks that every mistake is caught by at least one pin.

The definition: the SparseFlashMlaSoftmaxL1Norm article, section 三阶段计算公式
(stage 1 gather, stage 2 SimpleSoftmax against the forward LSE, stage 3
ReduceSum over the head group divided by G), and its constraints section for
mask_mode 3 (rightDownCausal).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked.json")
D = 512


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _ev(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "exp": math.exp, "log": math.log}))


def _bits(x: np.ndarray, dtype="bf16") -> np.ndarray:
    return W.bf16_bits_from_f32(x.astype(np.float32)) if dtype == "bf16" else \
        x.astype(np.float16).view(np.uint16)


def _close(a, b, rtol=2e-7, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    bad = ~(np.abs(a - b) <= atol + rtol * np.abs(b))
    assert not bad.any(), f"{what}: max |diff| {np.max(np.abs(a - b))}\n{a}\n{b}"


# ----------------------------------------------------------------------------
# hand-worked cases (closed forms, tests/golden/hand_worked.json)
# ----------------------------------------------------------------------------
def hand_sparse_inputs(topk4=False):
    rng = np.random.Generator(np.random.PCG64(11))
    k = rng.standard_normal((1, 8, 1, D)).astype(np.float32)
    for row, (a, b) in {5: (0.0, 1.0), 2: (1.0, 1.0), 7: (2.0, 1.0)}.items():
        k[0, row, 0, :] = 0.0
        k[0, row, 0, 0] = a
        k[0, row, 0, 1] = b
    q = np.zeros((1, 1, 2, D), dtype=np.float32)
    q[0, 0, 0, 0] = 1.0
    q[0, 0, 1, 0] = -1.0
    q[0, 0, 1, 1] = 2.0
    idx = np.array([5, 2, 7, -1] if topk4 else [5, 2, 7], dtype=np.int32).reshape(1, 1, 1, -1)
    tl = np.array([3], dtype=np.int32).reshape(1, 1, 1) if topk4 else None
    return _bits(q), _bits(k), idx, tl


def pin_hand_sparse(o):
    g = _golden()
    qb, kb, idx, _ = hand_sparse_inputs()
    lse = o.softmax_lse(qb, kb, dtype="bf16", sparse_indices=idx, softmax_scale=1.0)
    _close(lse[0], [_ev(x) for x in g["sparse_g2_topk3"]["lse"]], rtol=1e-12, what="hand lse")
    lse32 = lse.astype(np.float32).reshape(1, 1, 1, 2)
    out = o.softmax_l1_norm(qb, kb, lse32, dtype="bf16", sparse_indices=idx, softmax_scale=1.0)
    assert out.shape == (1, 1, 1, 3) and out.dtype == np.float32
    _close(out.reshape(-1), [_ev(x) for x in g["sparse_g2_topk3"]["out"]], what="hand out")
    # padded variant: slot 3 is padding (index -1, topk_length 3)
    qb, kb, idx, tl = hand_sparse_inputs(topk4=True)
    out = o.softmax_l1_norm(qb, kb, lse32, dtype="bf16", sparse_indices=idx, topk_length=tl,
                            softmax_scale=1.0)
    _close(out.reshape(-1), [_ev(x) for x in g["sparse_g2_topk4_padded"]["out"]], what="padded")
    assert out.reshape(-1)[3] == 0.0
    # topk_length 2 drops slot 2 (key 7) even though its index is valid
    out2 = o.softmax_l1_norm(qb, kb, lse32, dtype="bf16", sparse_indices=idx,
                             topk_length=np.array([2], dtype=np.int32).reshape(1, 1, 1),
                             softmax_scale=1.0)
    want = [_ev(x) for x in g["sparse_g2_topk4_padded"]["out"]]
    want[2] = 0.0
    _close(out2.reshape(-1), want, what="topk_length=2")


def _hand_dense(S1, S2, keyvals):
    k = np.zeros((1, S2, 1, D), dtype=np.float32)
    for j, v in enumerate(keyvals):
        k[0, j, 0, 0] = v
    q = np.zeros((1, S1, 1, D), dtype=np.float32)
    q[0, :, 0, 0] = 1.0
    return _bits(q), _bits(k)


def pin_hand_causal(o):
    g = _golden()
    # S1=2 < S2=3, scale 1/2
    qb, kb = _hand_dense(2, 3, [0.0, 1.0, 2.0])
    case = g["dense_causal_s1_2_s2_3"]
    lse = o.softmax_lse(qb, kb, dtype="bf16", softmax_scale=0.5, mask_mode=3)
    _close(lse[:, 0], [_ev(x) for x in case["lse"]], rtol=1e-12, what="causal lse")
    out = o.softmax_l1_norm(qb, kb, lse.astype(np.float32).reshape(1, 1, 2, 1), dtype="bf16",
                            softmax_scale=0.5, mask_mode=3)
    assert out.shape == (1, 2, 1, 3)
    _close(out.reshape(2, 3), [[_ev(x) for x in r] for r in case["out"]], what="causal out")
    # S1=3 > S2=2: the first row sees no key at all
    qb, kb = _hand_dense(3, 2, [0.0, 1.0])
    case = g["dense_causal_s1_3_s2_2"]
    lse = o.softmax_lse(qb, kb, dtype="bf16", softmax_scale=1.0, mask_mode=3)
    assert np.isneginf(lse[0, 0])
    out = o.softmax_l1_norm(qb, kb, lse.astype(np.float32).reshape(1, 1, 3, 1), dtype="bf16",
                            softmax_scale=1.0, mask_mode=3)
    _close(out.reshape(3, 2), [[_ev(x) for x in r] for r in case["out"]], what="causal S1>S2")
    assert np.all(out.reshape(3, 2)[0] == 0.0)


# ----------------------------------------------------------------------------
# random tiny workloads
# ----------------------------------------------------------------------------
def tiny_cases():
    """A spread of small seeded workloads: sparse/dense, BSND/TND, mask 0/3,
    bf16/fp16, G from 1 to 8, S1 above/below S2, ragged topk_length."""
    c = []
    c.append(W.make_workload(layout="BSND", dtype="bf16", B=2, S1=5, S2=9, G=3, topk=6,
                             mask_mode=3, seed=101, lse=None))
    c.append(W.make_workload(layout="BSND", dtype="fp16", B=1, S1=7, S2=5, G=2, topk=0,
                             mask_mode=3, seed=102, lse=None))
    c.append(W.make_workload(layout="BSND", dtype="bf16", B=1, S1=4, S2=12, G=5, topk=0,
                             mask_mode=0, seed=103, lse=None))
    c.append(W.make_workload(layout="TND", dtype="fp16", seqlens_q=[3, 6], seqlens_k=[5, 4],
                             G=4, topk=4, mask_mode=3, seed=104, lse=None))
    c.append(W.make_workload(layout="TND", dtype="bf16", seqlens_q=[4, 2], seqlens_k=[4, 7],
                             G=2, topk=0, mask_mode=3, seed=105, lse=None))
    c.append(W.make_workload(layout="BSND", dtype="bf16", B=1, S1=6, S2=10, G=1, topk=7,
                             mask_mode=0, seed=106, lse=None))
    # arbitrary indices: keys hidden by the causal mask, -1, and out-of-range
    # values, with no topk_length (every slot is a candidate)
    w = W.make_workload(layout="BSND", dtype="fp16", B=2, S1=6, S2=8, G=2, topk=10,
                        mask_mode=3, seed=107, lse=None, with_topk_length=False)
    rng = np.random.Generator(np.random.PCG64(107))
    w.sparse_indices = rng.integers(-2, 11, size=w.sparse_indices.shape).astype(np.int32)
    c.append(w)
    wt = W.make_workload(layout="TND", dtype="bf16", seqlens_q=[5, 3], seqlens_k=[4, 9],
                         G=3, topk=7, mask_mode=3, seed=108, lse=None, with_topk_length=False)
    wt.sparse_indices = rng.integers(-1, 11, size=wt.sparse_indices.shape).astype(np.int32)
    c.append(wt)
    return c


def kw(w):
    return dict(dtype=w.dtype, sparse_indices=w.sparse_indices, topk_length=w.topk_length,
                cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k,
                softmax_scale=w.softmax_scale, max_seqlen_k=w.max_seqlen_k,
                mask_mode=w.mask_mode, layout=w.layout)


def with_exact_lse(o, w):
    lse = o.softmax_lse(w.q_bits, w.k_bits, **kw(w))
    W.set_lse_rows(w, lse.astype(np.float32))
    return w


def pin_row_sums(o):
    """With the forward LSE over the same valid set, each head's P sums to 1
    over the valid slots, so the head mean does too; a row with no valid slot
    is all 0."""
    for w in tiny_cases():
        with_exact_lse(o, w)
        out = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w))
        rows = out.reshape(w.n_tokens, -1).astype(np.float64)
        lse = w.lse_rows()
        for t in range(w.n_tokens):
            s = rows[t].sum()
            if np.isneginf(lse[t, 0]):
                assert s == 0.0, f"{w.layout} row {t}: no valid slot but sum {s}"
            else:
                assert abs(s - 1.0) < 2e-6, f"{w.layout} row {t}: sum {s}"


def _valid_by_hand(w):
    """Validity table (n_tokens, width) written out from the constraints:
    key inside its sequence, slot below topk_length, causal j <= r + Sk - Sq."""
    tab = w.token_table()
    width = w.out_width
    V = np.zeros((w.n_tokens, width), dtype=bool)
    J = np.zeros((w.n_tokens, width), dtype=np.int64)
    for t in range(w.n_tokens):
        b, r, Sq, k0, Sk = (int(x) for x in tab[t])
        for i in range(width):
            if w.sparse_indices is not None:
                j = int(w.sparse_indices.reshape(w.n_tokens, -1)[t, i])
                if w.topk_length is not None and i >= int(w.topk_length.reshape(-1)[t]):
                    continue
            else:
                j = i
            if not (0 <= j < Sk):
                continue
            if w.mask_mode == 3 and not (j <= r + Sk - Sq):
                continue
            V[t, i] = True
            J[t, i] = k0 + j
    return V, J


def pin_g1_textbook_softmax(o):
    """G = 1: the operator is a plain softmax of scale * q.k over the valid
    slots (scipy.special.softmax), scaled by exp(true_lse - lse) when the LSE
    passed in is not the true one."""
    for w in tiny_cases():
        if w.G != 1:
            # rebuild the same geometry with one head
            w = W.make_workload(layout=w.layout, dtype=w.dtype, B=w.batch,
                                S1=w.max_seqlen_q, S2=max(w.seqlen_k_bsnd, 1),
                                seqlens_q=None if w.cu_seqlens_q is None else np.diff(w.cu_seqlens_q),
                                seqlens_k=None if w.cu_seqlens_k is None else np.diff(w.cu_seqlens_k),
                                G=1, topk=w.topk, mask_mode=w.mask_mode, seed=w.seed + 1000, lse=None)
        V, J = _valid_by_hand(w)
        qf = W.half_bits_to_f32(w.q_bits, w.dtype).astype(np.float64).reshape(w.n_tokens, -1)
        kf = W.half_bits_to_f32(w.k_bits, w.dtype).astype(np.float64).reshape(-1, qf.shape[1])
        rng = np.random.Generator(np.random.PCG64(7))
        shift = rng.uniform(-0.5, 0.5, size=w.n_tokens)
        lse_in = np.zeros(w.n_tokens)
        want = np.zeros((w.n_tokens, w.out_width))
        for t in range(w.n_tokens):
            v = np.flatnonzero(V[t])
            if len(v) == 0:
                lse_in[t] = -np.inf
                continue
            x = w.softmax_scale * (kf[J[t, v]] @ qf[t])
            true_lse = scipy.special.logsumexp(x)
            lse_in[t] = np.float32(true_lse + shift[t])
            want[t, v] = scipy.special.softmax(x) * np.exp(true_lse - lse_in[t])
        W.set_lse_rows(w, lse_in.astype(np.float32)[:, None])
        out = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w))
        _close(out.reshape(w.n_tokens, -1), want, rtol=1e-6, atol=1e-12, what="G=1 softmax")


def pin_brute_force(o):
    """Every output element from explicit Python loops over slots, heads and
    the 512 products (no matrix routine), on the tiny workloads."""
    for w in tiny_cases():
        rng = np.random.Generator(np.random.PCG64(w.seed))
        lse_rows = rng.uniform(0.5, 3.0, size=(w.n_tokens, w.G)).astype(np.float32)
        W.set_lse_rows(w, lse_rows)
        V, J = _valid_by_hand(w)
        qf = W.half_bits_to_f32(w.q_bits, w.dtype).reshape(w.n_tokens, w.G, -1).tolist()
        kf = W.half_bits_to_f32(w.k_bits, w.dtype).reshape(-1, D).tolist()
        want = np.zeros((w.n_tokens, w.out_width))
        for t in range(w.n_tokens):
            for i in range(w.out_width):
                if not V[t, i]:
                    continue
                krow = kf[J[t, i]]
                acc = 0.0
                for g in range(w.G):
                    qrow = qf[t][g]
                    dot = 0.0
                    for d in range(D):
                        dot += qrow[d] * krow[d]
                    acc += math.exp(w.softmax_scale * dot - float(lse_rows[t, g]))
                want[t, i] = acc / w.G
        out = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w))
        _close(out.reshape(w.n_tokens, -1), want, rtol=2e-7, atol=1e-30, what="brute force")


def pin_lse_logsumexp(o):
    """softmax_lse equals scipy.special.logsumexp of scale * q.k over the
    valid set written out by hand (every head separately), and -inf for a row
    with no valid slot.  One extra case draws topk_length below the number of
    valid indices, so that it cuts real keys."""
    cut = W.make_workload(layout="BSND", dtype="bf16", B=2, S1=6, S2=12, G=3, topk=8, mask_mode=0,
                          seed=109, lse=None)
    rng = np.random.Generator(np.random.PCG64(109))
    cut.topk_length = rng.integers(0, 9, size=cut.topk_length.shape).astype(np.int32)
    for w in tiny_cases() + [cut]:
        V, J = _valid_by_hand(w)
        qf = W.half_bits_to_f32(w.q_bits, w.dtype).astype(np.float64).reshape(w.n_tokens, w.G, -1)
        kf = W.half_bits_to_f32(w.k_bits, w.dtype).astype(np.float64).reshape(-1, qf.shape[2])
        got = o.softmax_lse(w.q_bits, w.k_bits, **kw(w))
        assert got.shape == (w.n_tokens, w.G)
        for t in range(w.n_tokens):
            v = np.flatnonzero(V[t])
            if len(v) == 0:
                assert np.all(np.isneginf(got[t])), f"row {t}: no valid slot, lse {got[t]}"
                continue
            x = w.softmax_scale * (qf[t] @ kf[J[t, v]].T)          # (G, n)
            _close(got[t], scipy.special.logsumexp(x, axis=1), rtol=1e-12, what="lse logsumexp")


def pin_sparse_equals_dense(o):
    """Selecting every visible key in ascending order makes the sparse form
    equal the dense form column for column; a random selection, scattered back
    by index, equals the dense form with the unselected keys masked out
    (their exp taken as 0) under the same LSE."""
    for layout, seq in (("BSND", None), ("TND", ([5, 3], [6, 4]))):
        dense = W.make_workload(layout=layout, dtype="bf16", B=2, S1=5, S2=6,
                                seqlens_q=None if seq is None else seq[0],
                                seqlens_k=None if seq is None else seq[1],
                                G=3, topk=0, mask_mode=3, seed=200, lse=None)
        with_exact_lse(o, dense)
        d_out = o.softmax_l1_norm(dense.q_bits, dense.k_bits, dense.softmax_lse, **kw(dense))
        d_rows = d_out.reshape(dense.n_tokens, -1)
        tab = dense.token_table()
        width = dense.out_width
        idx = np.full((dense.n_tokens, width), -1, dtype=np.int32)
        tl = np.zeros(dense.n_tokens, dtype=np.int32)
        for t in range(dense.n_tokens):
            b, r, Sq, k0, Sk = (int(x) for x in tab[t])
            vis = [j for j in range(Sk) if j <= r + Sk - Sq]
            idx[t, :len(vis)] = vis
            tl[t] = len(vis)
        lead = dense.q_bits.shape[:-2]
        s_out = o.softmax_l1_norm(dense.q_bits, dense.k_bits, dense.softmax_lse,
                                  **{**kw(dense), "sparse_indices": idx.reshape(*lead, 1, width),
                                     "topk_length": tl.reshape(*lead, 1)})
        s_rows = s_out.reshape(dense.n_tokens, -1)
        assert np.array_equal(s_rows, d_rows), f"{layout}: ascending-all sparse != dense"
        # random subset: scatter back by index and compare with a masked dense softmax
        rng = np.random.Generator(np.random.PCG64(201))
        qf = W.half_bits_to_f32(dense.q_bits, "bf16").astype(np.float64).reshape(dense.n_tokens, 3, D)
        kf = W.half_bits_to_f32(dense.k_bits, "bf16").astype(np.float64).reshape(-1, D)
        lse = dense.lse_rows().astype(np.float64)
        for t in range(dense.n_tokens):
            b, r, Sq, k0, Sk = (int(x) for x in tab[t])
            vis = [j for j in range(Sk) if j <= r + Sk - Sq]
            if not vis:
                continue
            pick = rng.permutation(vis)[: max(1, len(vis) // 2)]
            one = o.softmax_l1_norm_rows(dense.q_bits, dense.k_bits, dense.softmax_lse, [t],
                                         **{**kw(dense), "sparse_indices":
                                            np.pad(pick, (0, width - len(pick)), constant_values=-1)
                                            .reshape(1, width).repeat(dense.n_tokens, 0)
                                            .reshape(*lead, 1, width).astype(np.int32)})[0]
            scat = np.zeros(width)
            scat[pick] = one[: len(pick)]
            logits = np.full((3, width), -np.inf)
            logits[:, pick] = dense.softmax_scale * (qf[t] @ kf[k0 + pick].T)
            want = np.exp(logits - lse[t][:, None]).mean(axis=0)
            _close(scat, want, rtol=2e-7, what=f"{layout} scattered subset")


def pin_layout_equivalence(o):
    """A TND batch equals each of its sequences run alone as BSND with B = 1."""
    w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[4, 2, 5], seqlens_k=[6, 3, 5],
                        G=2, topk=5, mask_mode=3, seed=300, lse=None)
    with_exact_lse(o, w)
    out = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w)).reshape(w.n_tokens, -1)
    for b, q0, Sq, k0, Sk in w.sequences():
        qb = w.q_bits[q0:q0 + Sq].reshape(1, Sq, w.G, D)
        kb = w.k_bits[k0:k0 + Sk].reshape(1, Sk, 1, D)
        ib = w.sparse_indices[q0:q0 + Sq].reshape(1, Sq, 1, -1)
        tb = w.topk_length[q0:q0 + Sq].reshape(1, Sq, 1)
        lb = w.lse_rows()[q0:q0 + Sq].reshape(1, 1, Sq, w.G)
        o_b = o.softmax_l1_norm(qb, kb, lb, dtype="fp16", sparse_indices=ib, topk_length=tb,
                                softmax_scale=w.softmax_scale, mask_mode=3, layout="BSND")
        assert np.array_equal(o_b.reshape(Sq, -1), out[q0:q0 + Sq]), f"sequence {b}"


def pin_head_symmetries(o):
    """Identical heads give one head's softmax; permuting the slots permutes
    the output; permuting the heads (with their LSE) changes nothing."""
    w = W.make_workload(layout="BSND", dtype="bf16", B=1, S1=4, S2=16, G=4, topk=8,
                        mask_mode=0, seed=400, lse=None)
    q = w.q_bits.copy()
    q[:, :, 1:, :] = q[:, :, :1, :]
    w1 = W.Workload(**{**w.__dict__, "q_bits": q})
    with_exact_lse(o, w1)
    out4 = o.softmax_l1_norm(w1.q_bits, w1.k_bits, w1.softmax_lse, **kw(w1))
    w2 = W.Workload(**{**w1.__dict__, "q_bits": q[:, :, :1, :].copy(), "G": 1,
                       "softmax_lse": w1.softmax_lse[..., :1].copy()})
    out1 = o.softmax_l1_norm(w2.q_bits, w2.k_bits, w2.softmax_lse, **kw(w2))
    _close(out4, out1, rtol=2e-7, what="identical heads")
    with_exact_lse(o, w)
    base = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w)).reshape(4, -1)
    perm = np.random.Generator(np.random.PCG64(401)).permutation(8)
    wp = W.Workload(**{**w.__dict__, "sparse_indices": w.sparse_indices[..., perm].copy()})
    outp = o.softmax_l1_norm(wp.q_bits, wp.k_bits, wp.softmax_lse, **kw(wp)).reshape(4, -1)
    _close(outp, base[:, perm], rtol=2e-7, what="slot permutation")
    hp = np.array([2, 0, 3, 1])
    wh = W.Workload(**{**w.__dict__, "q_bits": w.q_bits[:, :, hp, :].copy(),
                       "softmax_lse": w.softmax_lse[..., hp].copy()})
    outh = o.softmax_l1_norm(wh.q_bits, wh.k_bits, wh.softmax_lse, **kw(wh)).reshape(4, -1)
    _close(outh, base, rtol=2e-7, what="head permutation")


def pin_seqused_truncation(o):
    """seqused_q / seqused_k (reading R11) equal running the operator on the
    truncated sequences -- the first seqused_q queries and first seqused_k
    keys of each batch entry, packed as TND -- with the dropped query rows 0;
    seqused equal to the full lengths changes nothing."""
    cases = [
        dict(layout="BSND", dtype="bf16", B=3, S1=9, S2=12, G=3, topk=7, mask_mode=3, seed=500),
        dict(layout="BSND", dtype="fp16", B=2, S1=8, S2=10, G=2, topk=0, mask_mode=3, seed=501),
        dict(layout="TND", dtype="bf16", seqlens_q=[6, 9], seqlens_k=[8, 9], G=2, topk=6, mask_mode=3, seed=502),
        dict(layout="TND", dtype="fp16", seqlens_q=[5, 7], seqlens_k=[9, 7], G=4, topk=0, mask_mode=0, seed=503),
    ]
    for ci, case in enumerate(cases):
        w = W.make_workload(lse=None, **case)
        rng = np.random.Generator(np.random.PCG64(600 + ci))
        W.set_lse_rows(w, rng.uniform(0.5, 3.0, size=(w.n_tokens, w.G)).astype(np.float32))
        seqs = list(w.sequences())
        su_q = np.array([int(rng.integers(0, Sq + 2)) for (_, _, Sq, _, _) in seqs], dtype=np.int32)
        su_k = np.array([int(rng.integers(0, Sk + 2)) for (_, _, _, _, Sk) in seqs], dtype=np.int32)
        full_q = np.array([Sq for (_, _, Sq, _, _) in seqs], dtype=np.int32)
        full_k = np.array([Sk for (_, _, _, _, Sk) in seqs], dtype=np.int32)
        base = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w)).reshape(w.n_tokens, -1)
        same = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, seqused_q=full_q, seqused_k=full_k,
                                 **kw(w)).reshape(w.n_tokens, -1)
        assert np.array_equal(base, same), "seqused = full lengths must change nothing"
        got = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, seqused_q=su_q, seqused_k=su_k,
                                **kw(w)).reshape(w.n_tokens, -1)
        width = w.out_width
        lse_rows = w.lse_rows()
        lse_cut = o.softmax_lse(w.q_bits, w.k_bits, seqused_q=su_q, seqused_k=su_k, **kw(w))
        for b, q0, Sq, k0, Sk in seqs:
            sq, sk = min(Sq, int(su_q[b])), min(Sk, int(su_k[b]))
            assert np.all(got[q0 + sq:q0 + Sq] == 0.0), f"case {ci} seq {b}: unused rows must be 0"
            if sq == 0:
                continue
            qb = w.q_bits.reshape(w.n_tokens, w.G, D)[q0:q0 + sq]
            kb = w.k_bits.reshape(-1, 1, D)[k0:k0 + sk] if sk > 0 else np.zeros((0, 1, D), np.uint16)
            sub = dict(dtype=w.dtype, softmax_scale=w.softmax_scale, mask_mode=w.mask_mode, layout="TND",
                       cu_seqlens_q=np.array([0, sq], np.int32), cu_seqlens_k=np.array([0, sk], np.int32),
                       max_seqlen_k=width)
            if w.sparse_indices is not None:
                sub["sparse_indices"] = w.sparse_indices.reshape(w.n_tokens, 1, -1)[q0:q0 + sq]
                if w.topk_length is not None:
                    sub["topk_length"] = w.topk_length.reshape(w.n_tokens, 1)[q0:q0 + sq]
            want = o.softmax_l1_norm(qb, kb, lse_rows[q0:q0 + sq].reshape(1, sq, w.G), **sub).reshape(sq, -1)
            assert np.array_equal(got[q0:q0 + sq], want), f"case {ci} seq {b}: truncated run differs"
            lse_want = o.softmax_lse(qb, kb, **sub)
            assert np.array_equal(lse_cut[q0:q0 + sq], lse_want), f"case {ci} seq {b}: truncated lse differs"
        for b, q0, Sq, k0, Sk in seqs:
            sq = min(Sq, int(su_q[b]))
            assert np.all(np.isneginf(lse_cut[q0 + sq:q0 + Sq])), f"case {ci} seq {b}: unused rows' lse"


def _expand_compressed(w, c, res):
    """The compressed workload ``w`` (TND) restated on original positions:
    sequence b gets L_b = Sk_b*c + res_b key rows, compressed key j sits at
    position j*c + c - 1 (the other rows are zero and never selected), and
    every index j in [0, Sk_b) becomes j*c + c - 1 (-1 stays -1; indices past
    the sequence stay past it).  Returns (k_bits, sparse_indices, cu_seqlens_k)."""
    seqs = list(w.sequences())
    kv = w.k_bits.reshape(-1, D)
    rows, cu = [], [0]
    for b, q0, Sq, k0, Sk in seqs:
        L = Sk * c + int(res[b])
        kb = np.zeros((L, D), np.uint16)
        if Sk:
            kb[np.arange(Sk) * c + c - 1] = kv[k0:k0 + Sk]
        rows.append(kb)
        cu.append(cu[-1] + L)
    k_exp = np.concatenate(rows).reshape(-1, 1, D) if rows else np.zeros((0, 1, D), np.uint16)
    if w.sparse_indices is not None:
        idx = w.sparse_indices.reshape(w.n_tokens, -1).astype(np.int64)
        tab = w.token_table()
        Sk_t = tab[:, 4:5]
        L_t = np.array([Sk * c + int(res[b]) for (b, _, _, _, Sk) in seqs])[tab[:, 0]][:, None]
        inside = (idx >= 0) & (idx < Sk_t)
        idx_exp = np.where(inside, idx * c + c - 1, np.where(idx < 0, idx, L_t + idx))
    else:
        width = w.out_width
        idx_exp = np.tile(np.arange(width) * c + c - 1, (w.n_tokens, 1))
        tab = w.token_table()
        idx_exp = np.where(np.arange(width)[None, :] < tab[:, 4:5], idx_exp, -1)
    return k_exp, idx_exp.astype(np.int32).reshape(w.n_tokens, 1, -1), np.array(cu, np.int32)


def pin_compressed_keys(o):
    """Compressed keys (reading R12: key j covers original positions j*c ..
    j*c + c - 1 of L = Sk*c + cmp_residual_k positions; mask 3 keeps a key
    when its whole block is visible)."""
    g = _golden()
    qb, kb = _hand_dense(2, 3, [0.0, 1.0, 2.0])
    for res, name in ((0, "compressed_dense_r4_res0"), (1, "compressed_dense_r4_res1")):
        case = g[name]
        cr = np.array([res], np.int32)
        lse = o.softmax_lse(qb, kb, dtype="bf16", softmax_scale=1.0, mask_mode=3, cmp_ratio=4, cmp_residual_k=cr)
        _close(lse[:, 0], [_ev(x) for x in case["lse"]], rtol=1e-12, what=f"{name} lse")
        out = o.softmax_l1_norm(qb, kb, lse.astype(np.float32).reshape(1, 1, 2, 1), dtype="bf16",
                                softmax_scale=1.0, mask_mode=3, cmp_ratio=4, cmp_residual_k=cr)
        _close(out.reshape(2, 3), [[_ev(x) for x in r] for r in case["out"]], what=f"{name} out")
    qb12, _ = _hand_dense(12, 3, [0.0, 1.0, 2.0])
    lse = o.softmax_lse(qb12, kb, dtype="bf16", softmax_scale=1.0, mask_mode=3, cmp_ratio=4,
                        cmp_residual_k=np.array([0], np.int32))
    out = o.softmax_l1_norm(qb12, kb, np.where(np.isneginf(lse), 0, lse).astype(np.float32).reshape(1, 1, 12, 1),
                            dtype="bf16", softmax_scale=1.0, mask_mode=3, cmp_ratio=4,
                            cmp_residual_k=np.array([0], np.int32)).reshape(12, 3)
    assert list((out != 0).sum(axis=1)) == g["compressed_dense_r4_s1_12"]["visible"]
    assert np.all(np.isneginf(lse[:3, 0])) and np.all(np.isfinite(lse[3:, 0]))

    # ratio 1 (residual 0) is the operator without compression; with mask 0
    # neither the ratio nor the residual matters
    for w in tiny_cases():
        with_exact_lse(o, w)
        base = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, **kw(w))
        zeros = np.zeros(w.batch, np.int32)
        assert np.array_equal(base, o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, cmp_ratio=1,
                                                      cmp_residual_k=zeros, **kw(w)))
        if w.mask_mode == 0:
            other = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, cmp_ratio=16,
                                      cmp_residual_k=np.full(w.batch, 7, np.int32), **kw(w))
            assert np.array_equal(base, other), "mask 0 must not depend on the compression"

    # the compressed operator equals the uncompressed one on the original
    # positions, with each compressed key at the end of its block
    cases = [
        dict(layout="TND", dtype="bf16", seqlens_q=[5, 9, 3], seqlens_k=[7, 4, 6], G=3, topk=5, mask_mode=3,
             seed=800, c=4, res=[1, 3, 0]),
        dict(layout="TND", dtype="fp16", seqlens_q=[6, 2], seqlens_k=[5, 9], G=2, topk=0, mask_mode=3,
             seed=801, c=3, res=[2, 0], max_seqlen_k=10),
        dict(layout="TND", dtype="bf16", seqlens_q=[40], seqlens_k=[3], G=2, topk=0, mask_mode=3,
             seed=802, c=16, res=[5]),
    ]
    for case in cases:
        c, res = case.pop("c"), np.array(case.pop("res"), np.int32)
        w = W.make_workload(lse=None, **case)
        rng = np.random.Generator(np.random.PCG64(case["seed"]))
        W.set_lse_rows(w, rng.uniform(0.5, 3.0, size=(w.n_tokens, w.G)).astype(np.float32))
        if w.sparse_indices is not None:
            w.sparse_indices = rng.integers(-2, max(w.k_bits.shape[0], 2) + 1,
                                            size=w.sparse_indices.shape).astype(np.int32)
        got = o.softmax_l1_norm(w.q_bits, w.k_bits, w.softmax_lse, cmp_ratio=c, cmp_residual_k=res, **kw(w))
        lse_c = o.softmax_lse(w.q_bits, w.k_bits, cmp_ratio=c, cmp_residual_k=res, **kw(w))
        k_exp, idx_exp, cu_k = _expand_compressed(w, c, res)
        sub = dict(dtype=w.dtype, softmax_scale=w.softmax_scale, mask_mode=w.mask_mode, layout="TND",
                   cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=cu_k, sparse_indices=idx_exp,
                   topk_length=w.topk_length, max_seqlen_k=int(np.diff(cu_k).max()))
        want = o.softmax_l1_norm(w.q_bits, k_exp, w.softmax_lse, **sub).reshape(w.n_tokens, -1)
        assert np.array_equal(got.reshape(w.n_tokens, -1), want[:, :got.reshape(w.n_tokens, -1).shape[1]]), \
            f"compressed case {case['seed']} differs from its expansion"
        assert np.array_equal(lse_c, o.softmax_lse(w.q_bits, k_exp, **sub)), f"lse of case {case['seed']}"

    # the article's TND call: 16 queries, 2048 compressed keys of ratio 128,
    # residual 0, right-down causal, dense: output (T1, 1, 2048); query r
    # keeps floor((r + 2048*128 - 16 + 1) / 128) keys (row 0 misses the last
    # block, which holds later positions; row 15 keeps all 2048)
    w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[16], seqlens_k=[2048], G=2, topk=0, mask_mode=3,
                        seed=803, lse=None)
    kwc = dict(kw(w), cmp_ratio=128, cmp_residual_k=np.zeros(1, np.int32))
    lse = o.softmax_lse(w.q_bits, w.k_bits, **kwc)
    out = o.softmax_l1_norm(w.q_bits, w.k_bits, lse.astype(np.float32).reshape(1, 16, 2), **kwc)
    assert out.shape == (16, 1, 2048) and np.all(np.isfinite(out))
    kept = (out.reshape(16, 2048) != 0).sum(axis=1)
    assert list(kept) == [min(2048, (r + 2048 * 128 - 16 + 1) // 128) for r in range(16)]
    assert kept[0] == 2047 and kept[15] == 2048


ALL_PINS = [pin_hand_sparse, pin_hand_causal, pin_row_sums, pin_g1_textbook_softmax,
            pin_brute_force, pin_sparse_equals_dense, pin_layout_equivalence,
            pin_head_symmetries, pin_seqused_truncation, pin_lse_logsumexp, pin_compressed_keys]
