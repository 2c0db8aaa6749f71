"""The seeded generators: shapes, index structure and determinism (no GPU)."""
import numpy as np

import workloads as W


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, 1.0 + 2**-9, -2.5e-3, 3.0e38], dtype=np.float32)
    bits = W.bf16_bits_from_f32(x)
    back = W.half_bits_to_f32(bits, "bf16")
    # 1+2^-9 is a tie between 1 and 1+2^-7... ties go to the even mantissa (1.0)
    assert back[0] == 1.0 and back[3] == 1.0
    assert back[2] == np.float32(1.0 + 2**-7)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2**-8)


def test_determinism_and_seed_sensitivity():
    a = W.make_workload(B=1, S1=8, S2=64, G=4, topk=16, mask_mode=3, seed=9)
    b = W.make_workload(B=1, S1=8, S2=64, G=4, topk=16, mask_mode=3, seed=9)
    c = W.make_workload(B=1, S1=8, S2=64, G=4, topk=16, mask_mode=3, seed=10)
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.sparse_indices, b.sparse_indices)
    assert not np.array_equal(a.q_bits, c.q_bits)


def test_uniform_visible_indices():
    w = W.make_workload(B=2, S1=40, S2=40, G=2, topk=16, mask_mode=3, seed=5)
    idx = w.sparse_indices.reshape(w.n_tokens, -1)
    tl = w.topk_length.reshape(-1)
    tab = w.token_table()
    for t in range(w.n_tokens):
        r = tab[t, 1]
        n = int(tl[t])
        assert n == min(16, r + 1)
        sel = idx[t, :n]
        assert len(np.unique(sel)) == n and sel.min() >= 0 and sel.max() <= r
        assert np.all(idx[t, n:] == -1)


def test_clustered_indices_structure():
    w = W.make_workload(B=1, S1=3000, S2=3000, G=1, topk=2048, mask_mode=3,
                        index_mode="clustered", seed=5, lse=None)
    idx = w.sparse_indices.reshape(w.n_tokens, -1)
    for t in (0, 100, 2047, 2048, 2600, 2999):
        n = min(2048, t + 1)
        row = idx[t, :n]
        assert np.all(np.diff(row) > 0), "sorted, distinct"
        assert row[0] >= 0 and row[-1] == t
        if t + 1 > 2048:
            assert np.array_equal(row[-512:], np.arange(t - 511, t + 1)), "trailing window"


def test_config_geometry():
    w = W.make_config(1)
    assert w.q_bits.shape == (1, 16, 8, 512) and w.out_shape() == (1, 16, 1, 32)
    assert w.valid_slot_count() == 16 * 32
    w = W.make_config(2)
    assert w.out_shape() == (2, 512, 1, 512) and w.sparse_indices is None
    assert w.valid_slot_count() == 2 * 512 * 513 // 2


def test_oracle_pool_equals_direct_oracle_calls(tmp_path):
    """The process-pool helper of the full-size parity test returns exactly
    what the oracle's functions return when called directly."""
    import oracle
    import oracle_pool
    w = W.make_workload(layout="TND", dtype="fp16", seqlens_q=[5, 0, 9], seqlens_k=[40, 3, 300], G=4,
                        topk=64, mask_mode=3, seed=77)
    rows = [13, 0, 4, 5]
    lse, out = oracle_pool.lse_and_rows(w, rows, str(tmp_path / "w"), processes=2, chunk=3)
    kw = dict(dtype=w.dtype, sparse_indices=w.sparse_indices, topk_length=w.topk_length,
              cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k, softmax_scale=w.softmax_scale,
              max_seqlen_k=w.max_seqlen_k, mask_mode=w.mask_mode, layout=w.layout)
    lse_d = oracle.softmax_lse(w.q_bits, w.k_bits, rows=rows, **kw).astype(np.float32)
    assert np.array_equal(lse, lse_d)
    full = np.zeros((w.n_tokens, w.G), np.float32)
    full[rows] = lse_d
    assert np.array_equal(out, oracle.softmax_l1_norm_rows(w.q_bits, w.k_bits, full, rows, **kw))
