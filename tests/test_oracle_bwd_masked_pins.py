"""Pins for the oracle's masked backward (band / prefix masks, N_q != N_k):
reductions to the pinned square backward, central finite differences of the
forward's loss sum(dO o O) in every direction tried, D = rowsum(dO o O) from
the pinned masked forward, zero gradients where nothing is seen, and the
16-bit entry equal to the float64 one on widened inputs.  CPU only."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_fa2_gb300 import synthetic as sy


def _bits(B, H, Nq, Nk, d, dtype, seed):
    q = sy.make_qkv(B, H, Nq, d, dtype, seed)[0]
    _, k, v = sy.make_qkv(B, H, Nk, d, dtype, seed + 1)
    do = sy.make_qkv(B, H, Nq, d, dtype, seed + 2)[0]
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_square_masks_equal_the_pinned_backward(causal):
    q, k, v, do = _bits(2, 2, 29, 29, 8, sy.BF16, 61)
    wr = 0 if causal else -1
    a = oracle.attention_bwd_masked(q, k, v, do, sy.BF16, 0.4, window_left=-1, window_right=wr)
    b = oracle.attention_bwd(q, k, v, do, sy.BF16, 0.4, causal)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13, rtol=0)


MASKS = [(-1, -1, 0), (-1, 0, 0), (2, 1, 0), (0, 0, 0), (3, 0, 2), (-1, 0, 4), (1, -1, 0)]


@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", [(5, 5), (4, 7), (7, 4)])
def test_finite_differences(mask, Nq, Nk):
    wl, wr, pre = mask
    rng = np.random.default_rng(Nq * 31 + Nk + 7 * wl + 5 * pre)
    d, scale = 3, 0.7
    q = rng.standard_normal((1, 2, Nq, d))
    k = rng.standard_normal((1, 2, Nk, d))
    v = rng.standard_normal((1, 2, Nk, d))
    do = rng.standard_normal((1, 2, Nq, d))
    dq, dk, dv, _ = oracle.attention_bwd_masked_f64(q, k, v, do, scale, wl, wr, pre)

    def loss(q_, k_, v_):
        o, _ = oracle.attention_fwd_masked_f64(q_, k_, v_, scale, wl, wr, pre)
        return float((o * do).sum())

    eps = 1e-6
    for trial in range(3):
        tq, tk, tv = (rng.standard_normal(x.shape) for x in (q, k, v))
        fd = (loss(q + eps * tq, k + eps * tk, v + eps * tv) - loss(q - eps * tq, k - eps * tk, v - eps * tv)) / (2 * eps)
        an = float((dq * tq).sum() + (dk * tk).sum() + (dv * tv).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (trial, fd, an)


@pytest.mark.parametrize("mask", MASKS)
def test_delta_is_rowsum_of_dout_times_o(mask):
    wl, wr, pre = mask
    q, k, v, do = _bits(1, 2, 20, 33, 8, sy.FP16, 71)
    _, _, _, delta = oracle.attention_bwd_masked(q, k, v, do, sy.FP16, 0.5, wl, wr, pre)
    o, _ = oracle.attention_fwd_masked(q, k, v, sy.FP16, 0.5, wl, wr, pre)
    np.testing.assert_allclose(delta, (oracle.widen(do, sy.FP16) * o).sum(-1), atol=1e-12, rtol=0)


def test_unseen_rows_and_keys_have_zero_gradients():
    # causal with N_q > N_k: rows 0..5 see no key; window (1, 0) with N_q < N_k: keys 0..7 are seen by no row
    q, k, v, do = _bits(1, 1, 10, 4, 8, sy.FP16, 81)
    dq, _, _, delta = oracle.attention_bwd_masked(q, k, v, do, sy.FP16, 1.0, -1, 0)
    assert np.all(dq[0, 0, :6] == 0) and np.all(delta[0, 0, :6] == 0) and np.any(dq[0, 0, 6:] != 0)
    q, k, v, do = _bits(1, 1, 4, 12, 8, sy.FP16, 82)
    _, dk, dv, _ = oracle.attention_bwd_masked(q, k, v, do, sy.FP16, 1.0, 1, 0)
    assert np.all(dk[0, 0, :7] == 0) and np.all(dv[0, 0, :7] == 0) and np.any(dv[0, 0, 7:] != 0)


def test_sixteen_bit_entry_equals_float64_entry():
    q, k, v, do = _bits(1, 2, 9, 14, 8, sy.BF16, 91)
    a = oracle.attention_bwd_masked(q, k, v, do, sy.BF16, 0.3, 4, 2, 3)
    b = oracle.attention_bwd_masked_f64(*(oracle.widen(x, sy.BF16) for x in (q, k, v, do)), 0.3, 4, 2, 3)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
