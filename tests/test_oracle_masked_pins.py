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
