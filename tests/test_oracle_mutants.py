"""Plant plausible mistakes in a private copy of the oracle and check that
each one fails at least one pin (so the pins would catch the same mistake in
the real oracle).  Mistakes are planted only in the copy, on the CPU."""
import importlib.util
import os

import numpy as np
import pytest

import oracle_pins as P

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "oracle", "smla_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("smla_oracle_copy", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_drop_scale(m):
    orig = m.simple_softmax
    m.simple_softmax = lambda q, k, v, lse, scale: orig(q, k, v, lse, 1.0)


def _mut_sign(m):
    def f(q, k, v, lse, scale):
        x = (q @ k.T) * scale
        p = np.zeros_like(x)
        p[:, v] = np.exp(np.asarray(lse)[:, None] - x[:, v])
        return p
    m.simple_softmax = f


def _mut_sum_not_mean(m):
    m.reduce_sum_g_mean = lambda p: p.sum(axis=0)


def _mut_divide_by_slots(m):
    m.reduce_sum_g_mean = lambda p: p.sum(axis=0) / p.shape[1]


def _mut_causal_off_by_one(m):
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        ok = orig(j, r=r, Sq=Sq, Sk=Sk, mask_mode=0, topk_len=topk_len, **extra)
        if mask_mode == 3:
            ok &= j < (r + Sk - Sq)
        return ok
    m.slot_valid = f


def _mut_causal_top_left(m):
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        ok = orig(j, r=r, Sq=Sq, Sk=Sk, mask_mode=0, topk_len=topk_len, **extra)
        if mask_mode == 3:
            ok &= j <= r
        return ok
    m.slot_valid = f


def _mut_ignore_topk_length(m):
    orig = m.slot_valid
    m.slot_valid = lambda j, *, r, Sq, Sk, mask_mode, topk_len, **extra: orig(
        j, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=None)


def _mut_mask_on_slot(m):
    """causal test applied to the slot number instead of the key position"""
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        ok = orig(j, r=r, Sq=Sq, Sk=Sk, mask_mode=0, topk_len=topk_len, **extra)
        if mask_mode == 3:
            ok &= np.arange(len(j)) <= (r + Sk - Sq)
        return ok
    m.slot_valid = f


def _mut_lse_head_order(m):
    orig = m.simple_softmax
    m.simple_softmax = lambda q, k, v, lse, scale: orig(q, k, v, np.asarray(lse)[::-1], scale)


def _mut_tnd_key_offset(m):
    orig = m.token_geometry
    def f(*a, **k):
        return [(b, r, Sq, 0, Sk) for (b, r, Sq, k0, Sk) in orig(*a, **k)]
    m.token_geometry = f


def _mut_keep_out_of_range(m):
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        ok = orig(np.where(j >= Sk, 0, j), r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=topk_len)
        return ok
    m.slot_valid = f


def _mut_log2(m):
    def f(q, k, v, lse, scale):
        x = (q @ k.T) * scale
        p = np.zeros_like(x)
        p[:, v] = np.exp2(x[:, v] - np.asarray(lse)[:, None])
        return p
    m.simple_softmax = f


def _mut_lse_no_scale(m):
    orig = m.softmax_lse
    def f(*a, **k):
        k = dict(k)
        k["softmax_scale"] = 1.0
        return orig(*a, **k)
    m.softmax_lse = f


def _mut_seqused_q_ignored(m):
    orig = m._effective
    m._effective = lambda g, sq, sk: orig(g, None, sk)


def _mut_seqused_causal_full_lengths(m):
    """seqused applied to the masks but the causal offset kept on full lengths"""
    orig_valid = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        return orig_valid(j, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=topk_len, **extra)
    m.slot_valid = f
    orig_eff = m._effective
    def eff(g, sq, sk):
        b, r, Sq, k0, Sk = orig_eff(g, sq, sk)
        b0, r0, Sq0, k00, Sk0 = g
        return b, r, Sq0, k0, Sk       # keeps the full query length for the offset
    m._effective = eff


def _mut_lse_base2(m):
    """the forward LSE reported in base 2"""
    orig = m.softmax_lse
    m.softmax_lse = lambda *a, **k: orig(*a, **k) / np.log(2.0)


def _mut_lse_drops_topk_length(m):
    """the forward LSE taken over every slot, ignoring topk_length"""
    orig = m.softmax_lse
    def f(*a, **k):
        k = dict(k)
        k["topk_length"] = None
        return orig(*a, **k)
    m.softmax_lse = f


def _mut_lse_mask_off(m):
    """the forward LSE taken without the causal mask"""
    orig = m.softmax_lse
    def f(*a, **k):
        k = dict(k)
        k["mask_mode"] = 0
        return orig(*a, **k)
    m.softmax_lse = f


def _mut_bf16_read_as_fp16(m):
    """bf16 bit patterns decoded as IEEE binary16"""
    orig = m.decode_half
    m.decode_half = lambda bits, dtype: orig(bits, "fp16")


def _mut_minus_one_wraps(m):
    """index -1 taken as the last key of the sequence (negative indexing)"""
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, **extra):
        jj = np.where(j < 0, Sk - 1, j)
        return orig(jj, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=topk_len, **extra)
    m.slot_valid = f
    orig_terms = m._row_terms
    def terms(t, geo, qv, kv, dtype, sparse_indices, topk_length, width, mask_mode,
              seqused_q=None, seqused_k=None, *rest):
        q_row, sel_k, valid = orig_terms(t, geo, qv, kv, dtype, sparse_indices, topk_length, width,
                                         mask_mode, seqused_q, seqused_k, *rest)
        if sparse_indices is not None:
            b, r, Sq, k0, Sk = m._effective(geo[t], seqused_q, seqused_k)
            idx_row = np.asarray(sparse_indices).reshape(len(geo), -1)[t].astype(np.int64)
            neg = (idx_row < 0) & valid
            if neg.any() and Sk > 0:
                sel_k = sel_k.copy()
                sel_k[neg] = m.decode_half(kv[k0 + Sk - 1], dtype)
        return q_row, sel_k, valid
    m._row_terms = terms


def _mut_seqused_k_ignored(m):
    orig = m._effective
    m._effective = lambda g, sq, sk: orig(g, sq, None)


def _mut_slots_in_key_order(m):
    """sparse outputs written in ascending key order instead of slot order"""
    orig = m.slot_key_positions
    def f(idx_row, width):
        j = orig(idx_row, width)
        return np.sort(j) if idx_row is not None else j
    m.slot_key_positions = f


def _mut_cmp_block_start(m):
    """compressed keys kept when their block merely starts at a visible position"""
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, cmp_ratio=1, orig_len=None):
        ok = orig(j, r=r, Sq=Sq, Sk=Sk, mask_mode=0, topk_len=topk_len)
        if mask_mode == 3:
            L = Sk if orig_len is None else orig_len
            ok &= j * cmp_ratio <= r + L - Sq
        return ok
    m.slot_valid = f


def _mut_cmp_residual_ignored(m):
    """the original key length taken as Sk * cmp_ratio, without the residual"""
    m.original_key_length = lambda Sk, b, c, res: Sk * int(c)


def _mut_cmp_ratio_ignored(m):
    """compressed keys masked as if each stood for one original position"""
    orig = m.slot_valid
    def f(j, *, r, Sq, Sk, mask_mode, topk_len, cmp_ratio=1, orig_len=None):
        return orig(j, r=r, Sq=Sq, Sk=Sk, mask_mode=mask_mode, topk_len=topk_len)
    m.slot_valid = f


MUTANTS = [_mut_drop_scale, _mut_sign, _mut_sum_not_mean, _mut_divide_by_slots,
           _mut_causal_off_by_one, _mut_causal_top_left, _mut_ignore_topk_length,
           _mut_mask_on_slot, _mut_lse_head_order, _mut_tnd_key_offset,
           _mut_keep_out_of_range, _mut_log2, _mut_lse_no_scale, _mut_seqused_q_ignored,
           _mut_seqused_causal_full_lengths, _mut_lse_base2, _mut_lse_drops_topk_length,
           _mut_lse_mask_off, _mut_bf16_read_as_fp16, _mut_minus_one_wraps,
           _mut_seqused_k_ignored, _mut_slots_in_key_order, _mut_cmp_block_start,
           _mut_cmp_residual_ignored, _mut_cmp_ratio_ignored]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__[5:])
def test_mutant_is_caught(mutant):
    m = fresh_oracle()
    mutant(m)
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(m)
        except (AssertionError, IndexError) as e:
            # a wrong value, or a gather outside K that the mistake led to;
            # not a TypeError from a stale override of an oracle function
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"mutant {mutant.__name__} passed every pin"
