"""Pins for the band-mask / unequal-length forward of the oracle: reductions
to the pinned full and causal definitions, closed forms, the per-row
sub-problem rule, empty rows, and a 50-digit brute force.  CPU only."""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from exact_tiled_attention_fa2_gb300 import synthetic as sy


def _qkv(B, H, Nq, Nk, d, dtype, seed):
    q = sy.make_qkv(B, H, Nq, d, dtype, seed)[0]
    _, k, v = sy.make_qkv(B, H, Nk, d, dtype, seed + 1)
    return q, k, v


@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
def test_no_window_is_full_attention(dtype):
    q, k, v = _qkv(1, 2, 37, 37, 8, dtype, 1)
    a = oracle.attention_fwd_masked(q, k, v, dtype, 0.3)
    b = oracle.attention_fwd(q, k, v, dtype, 0.3, False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
def test_right_window_zero_is_causal(dtype):
    q, k, v = _qkv(2, 1, 29, 29, 8, dtype, 3)
    a = oracle.attention_fwd_masked(q, k, v, dtype, 0.5, window_left=-1, window_right=0)
    b = oracle.attention_fwd(q, k, v, dtype, 0.5, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("Nq,Nk", [(16, 16), (5, 16)])
def test_zero_width_window_selects_one_key(Nq, Nk):
    q, k, v = _qkv(1, 2, Nq, Nk, 4, sy.FP16, 5)
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.FP16, 0.7, window_left=0, window_right=0)
    Q, K, V = (oracle.widen(x, sy.FP16) for x in (q, k, v))
    off = Nk - Nq
    for i in range(Nq):
        np.testing.assert_array_equal(o[:, :, i], V[:, :, i + off])
        np.testing.assert_allclose(lse[:, :, i], 0.7 * (Q[:, :, i] * K[:, :, i + off]).sum(-1), atol=1e-14, rtol=0)


def _row_by_subproblem(q, k, v, dtype, scale, i, lo, hi):
    """Row i over keys [lo, hi] as the last row of an unmasked square problem."""
    n = hi - lo + 1
    qs = np.repeat(q[:, :, i:i + 1], n, axis=2)
    return oracle.attention_fwd(qs, k[:, :, lo:hi + 1].copy(), v[:, :, lo:hi + 1].copy(), dtype, scale, False)


@pytest.mark.parametrize("Nq,Nk,wl,wr", [(40, 40, 7, 3), (40, 40, 5, 0), (12, 40, -1, 0), (12, 40, 6, 2),
                                         (40, 40, -1, 9)])
def test_each_row_is_the_unmasked_problem_on_its_key_range(Nq, Nk, wl, wr):
    q, k, v = _qkv(1, 2, Nq, Nk, 6, sy.BF16, 7)
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.BF16, 0.4, window_left=wl, window_right=wr)
    off = Nk - Nq
    for i in range(Nq):
        lo = max(0, i + off - wl) if wl >= 0 else 0
        hi = min(Nk - 1, i + off + wr) if wr >= 0 else Nk - 1
        so, sl = _row_by_subproblem(q, k, v, sy.BF16, 0.4, i, lo, hi)
        np.testing.assert_allclose(o[:, :, i], so[:, :, -1], atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[:, :, i], sl[:, :, -1], atol=1e-14, rtol=0)


def test_rows_without_keys_are_zero_with_minus_inf_lse():
    q, k, v = _qkv(1, 1, 10, 4, 3, sy.FP16, 9)         # causal, Nq > Nk: rows 0..5 see nothing
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.FP16, 1.0, window_left=-1, window_right=0)
    assert np.all(o[0, 0, :6] == 0) and np.all(np.isneginf(lse[0, 0, :6]))
    assert np.isfinite(lse[0, 0, 6:]).all()
    V = oracle.widen(v, sy.FP16)
    np.testing.assert_array_equal(o[0, 0, 6], V[0, 0, 0])   # row 6 faces key 0 only


def test_brute_force_band():
    getcontext().prec = 50
    Nq, Nk, d, wl, wr, scale = 4, 7, 3, 2, 1, 0.9
    q, k, v = _qkv(1, 1, Nq, Nk, d, sy.FP16, 11)
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.FP16, scale, window_left=wl, window_right=wr)
    Q, K, V = (oracle.widen(x, sy.FP16)[0, 0] for x in (q, k, v))
    off = Nk - Nq
    for i in range(Nq):
        keys = [j for j in range(Nk) if i + off - wl <= j <= i + off + wr]
        ex = [(j, (Decimal(repr(scale)) * sum(Decimal(repr(float(Q[i, c]))) * Decimal(repr(float(K[j, c])))
                                             for c in range(d))).exp()) for j in keys]
        tot = sum(e for _, e in ex)
        for c in range(d):
            assert o[0, 0, i, c] == pytest.approx(float(sum(e * Decimal(repr(float(V[j, c]))) for j, e in ex) / tot),
                                                  abs=1e-13)
        assert lse[0, 0, i] == pytest.approx(float(tot.ln()), abs=1e-13)


# ---------------------------------------------------------------- prefix (prefix-LM) and sampled rows


def _row_over_keys(q, k, v, dtype, scale, i, keys):
    """Row i attending to exactly the key indices `keys`, as the last row of an
    unmasked square problem over those keys (pinned full-attention definition)."""
    keys = np.asarray(keys, dtype=np.int64)
    qs = np.repeat(q[:, :, i:i + 1], keys.size, axis=2)
    so, sl = oracle.attention_fwd(qs, np.ascontiguousarray(k[:, :, keys]), np.ascontiguousarray(v[:, :, keys]), dtype,
                                  scale, False)
    return so[:, :, -1], sl[:, :, -1]


@pytest.mark.parametrize("wl,wr", [(-1, 0), (3, 0), (0, 0), (2, 5)])
def test_prefix_covering_all_keys_is_full_attention(wl, wr):
    q, k, v = _qkv(1, 2, 23, 23, 8, sy.FP16, 11)
    a = oracle.attention_fwd_masked(q, k, v, sy.FP16, 0.3, window_left=wl, window_right=wr, prefix_len=23)
    b = oracle.attention_fwd(q, k, v, sy.FP16, 0.3, False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
def test_prefix_lm_splits_into_full_prefix_and_causal_rest(dtype):
    """Causal with prefix P (N_q = N_k = N): rows i < P see exactly keys [0, P)
    (full attention on the first P rows and keys); rows i >= P see [0, i]
    (the causal rows)."""
    N, P = 31, 9
    q, k, v = _qkv(2, 1, N, N, 8, dtype, 13)
    o, lse = oracle.attention_fwd_masked(q, k, v, dtype, 0.45, window_left=-1, window_right=0, prefix_len=P)
    fo, fl = oracle.attention_fwd(np.ascontiguousarray(q[:, :, :P]), np.ascontiguousarray(k[:, :, :P]),
                                  np.ascontiguousarray(v[:, :, :P]), dtype, 0.45, False)
    co, cl = oracle.attention_fwd(q, k, v, dtype, 0.45, True)
    np.testing.assert_allclose(o[:, :, :P], fo, atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse[:, :, :P], fl, atol=1e-14, rtol=0)
    np.testing.assert_array_equal(o[:, :, P:], co[:, :, P:])
    np.testing.assert_array_equal(lse[:, :, P:], cl[:, :, P:])


@pytest.mark.parametrize("Nq,Nk,wl,wr,P", [(20, 20, 2, 0, 3), (12, 30, 4, 1, 5), (30, 12, 1, 0, 2)])
def test_prefix_with_window_sees_the_union_of_both_key_sets(Nq, Nk, wl, wr, P):
    """A window that leaves a gap after the prefix: row i sees [0, P) plus its
    band, by the unmasked definition over exactly that key set."""
    q, k, v = _qkv(1, 2, Nq, Nk, 5, sy.BF16, 17)
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.BF16, 0.6, window_left=wl, window_right=wr, prefix_len=P)
    off = Nk - Nq
    for i in range(Nq):
        band = set(range(max(0, i + off - wl), min(Nk - 1, i + off + wr) + 1))
        keys = sorted(band | set(range(min(P, Nk))))
        ro, rl = _row_over_keys(q, k, v, sy.BF16, 0.6, i, keys)
        np.testing.assert_allclose(o[:, :, i], ro, atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[:, :, i], rl, atol=1e-14, rtol=0)


@pytest.mark.parametrize("Nq,Nk,wl,wr,P", [(40, 40, -1, -1, 0), (40, 40, -1, 0, 0), (50, 20, 6, 0, 0),
                                           (20, 50, 3, 2, 4), (33, 33, -1, 0, 10)])
def test_sampled_rows_equal_the_whole_problem(Nq, Nk, wl, wr, P):
    q, k, v = _qkv(2, 3, Nq, Nk, 8, sy.FP16, 19)
    o, lse = oracle.attention_fwd_masked(q, k, v, sy.FP16, 0.35, window_left=wl, window_right=wr, prefix_len=P)
    rng = np.random.default_rng(5)
    bh = rng.integers(0, 6, size=40)
    rows = rng.integers(0, Nq, size=40)
    so, sl = oracle.attention_rows_masked(q, k, v, sy.FP16, 0.35, bh, rows, window_left=wl, window_right=wr,
                                          prefix_len=P)
    np.testing.assert_array_equal(so, o.reshape(6, Nq, 8)[bh, rows])
    np.testing.assert_array_equal(sl, lse.reshape(6, Nq)[bh, rows])


def test_sampled_rows_reject_out_of_range_indices():
    q, k, v = _qkv(1, 1, 8, 8, 4, sy.FP16, 21)
    with pytest.raises(ValueError):
        oracle.attention_rows_masked(q, k, v, sy.FP16, 1.0, [0], [8])
    with pytest.raises(ValueError):
        oracle.attention_rows_masked(q, k, v, sy.FP16, 1.0, [1], [0])
    with pytest.raises(ValueError):
        oracle.attention_fwd_masked(q, k, v, sy.FP16, 1.0, prefix_len=-1)
