"""Pins for the backward oracle (gradients of the forward pass for an upstream
gradient dO): central finite differences of the forward oracle, the identity
D_i = rowsum(dP_i o P_i) = rowsum(dO_i o O_i) that FlashAttention V2 in depth
section 7.3 states, and invariants of the softmax Jacobian.  CPU only."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_fa2_gb300 import synthetic as sy


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attention_fwd_f64(q, k, v, scale, causal)
    return float((o * dout).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_differences(causal):
    B, H, N, d = 1, 2, 5, 3
    q, k, v, dout = (_rand((B, H, N, d), s) for s in (1, 2, 3, 4))
    scale = 0.7
    dq, dk, dv, _ = oracle.attention_bwd_f64(q, k, v, dout, scale, causal)
    h = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy()
            xp[idx] += h
            xm = x.copy()
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = _loss(args["q"], args["k"], args["v"], dout, scale, causal)
            args[name] = xm
            fm = _loss(args["q"], args["k"], args["v"], dout, scale, causal)
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, atol=2e-8, rtol=2e-7, err_msg="d" + name)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_equals_rowsum_of_dout_times_out(causal):
    B, H, N, d = 2, 2, 9, 4
    q, k, v, dout = (_rand((B, H, N, d), s) for s in (5, 6, 7, 8))
    _, _, _, delta = oracle.attention_bwd_f64(q, k, v, dout, 0.5, causal)
    o, _ = oracle.attention_fwd_f64(q, k, v, 0.5, causal)
    np.testing.assert_allclose(delta, (dout * o).sum(-1), atol=1e-12, rtol=0)


def test_single_key():
    q, k, v, dout = (_rand((1, 3, 1, 4), s) for s in (9, 10, 11, 12))
    dq, dk, dv, _ = oracle.attention_bwd_f64(q, k, v, dout, 0.9, False)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    np.testing.assert_allclose(dv, dout, atol=0, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_column_sums(causal):
    # rows of P sum to 1, so sum_j dV_j = sum_i dO_i; rows of dS sum to 0, so sum_j dK_j = 0
    B, H, N, d = 1, 2, 11, 5
    q, k, v, dout = (_rand((B, H, N, d), s) for s in (13, 14, 15, 16))
    dq, dk, dv, _ = oracle.attention_bwd_f64(q, k, v, dout, 0.4, causal)
    np.testing.assert_allclose(dv.sum(axis=2), dout.sum(axis=2), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12, rtol=0)


def test_constant_values_give_no_query_or_key_gradient():
    B, H, N, d = 1, 1, 7, 3
    q, k, dout = (_rand((B, H, N, d), s) for s in (17, 18, 19))
    v = np.broadcast_to(_rand((1, 1, 1, d), 20), (B, H, N, d)).copy()
    dq, dk, dv, _ = oracle.attention_bwd_f64(q, k, v, dout, 0.8, False)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)


def test_causal_last_key_sees_only_last_row():
    B, H, N, d = 1, 1, 6, 2
    q, k, v, dout = (_rand((B, H, N, d), s) for s in (21, 22, 23, 24))
    scale = 0.6
    dq, dk, dv, _ = oracle.attention_bwd_f64(q, k, v, dout, scale, True)
    s = scale * q[0, 0, -1] @ k[0, 0].T
    p_last = np.exp(s[-1] - s.max()) / np.exp(s - s.max()).sum()
    np.testing.assert_allclose(dv[0, 0, -1], p_last * dout[0, 0, -1], atol=1e-14, rtol=0)


def test_16bit_entry_equals_widened_f64_entry():
    q, k, v, dout = sy.make_qkv(1, 2, 17, 8, sy.BF16, 31) + (sy.make_qkv(1, 2, 17, 8, sy.BF16, 32)[0],)
    g16 = oracle.attention_bwd(q, k, v, dout, sy.BF16, 0.35, True)
    g64 = oracle.attention_bwd_f64(*(oracle.widen(x, sy.BF16) for x in (q, k, v, dout)), 0.35, True)
    for a, b in zip(g16, g64):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_the_full_backward(causal):
    # the sampled-row entry point runs the rows pass of the full backward for
    # the listed rows: dQ rows and D_i equal the full function's, bit for bit
    B, H, N, d = 2, 3, 37, 16
    q, k, v = sy.make_qkv(B, H, N, d, sy.FP16, 41)
    dout = sy.make_qkv(B, H, N, d, sy.FP16, 42)[0]
    dq, _, _, delta = oracle.attention_bwd(q, k, v, dout, sy.FP16, 0.25, causal)
    rng = np.random.default_rng(43)
    bh_idx = np.sort(rng.integers(0, B * H, size=40))
    row_idx = rng.integers(0, N, size=40)
    dq_rows, delta_rows = oracle.attention_bwd_rows(q, k, v, dout, sy.FP16, 0.25, causal, bh_idx, row_idx)
    np.testing.assert_array_equal(dq_rows, dq.reshape(B * H, N, d)[bh_idx, row_idx])
    np.testing.assert_array_equal(delta_rows, delta.reshape(B * H, N)[bh_idx, row_idx])


def test_sampled_rows_reject_out_of_range_indices():
    q, k, v = sy.make_qkv(1, 1, 8, 4, sy.FP16, 44)
    with pytest.raises(ValueError):
        oracle.attention_bwd_rows(q, k, v, q, sy.FP16, 0.5, False, np.array([1]), np.array([0]))
    with pytest.raises(ValueError):
        oracle.attention_bwd_rows(q, k, v, q, sy.FP16, 0.5, False, np.array([0]), np.array([8]))


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_keys_equal_the_full_backward(causal):
    # the sampled-key entry point runs the keys pass of the full backward for
    # the listed keys (over the rows that see them): dK and dV rows equal the
    # full function's, bit for bit
    B, H, N, d = 1, 3, 45, 16
    q, k, v = sy.make_qkv(B, H, N, d, sy.BF16, 51)
    dout = sy.make_qkv(B, H, N, d, sy.BF16, 52)[0]
    _, dk, dv, _ = oracle.attention_bwd(q, k, v, dout, sy.BF16, 0.3, causal)
    keys = np.array([44, 40, 31, 3, 0, 44])
    for bh in range(B * H):
        dk_rows, dv_rows = oracle.attention_bwd_keys(q, k, v, dout, sy.BF16, 0.3, causal, bh, keys)
        np.testing.assert_array_equal(dk_rows, dk.reshape(B * H, N, d)[bh, keys])
        np.testing.assert_array_equal(dv_rows, dv.reshape(B * H, N, d)[bh, keys])


def test_sampled_keys_reject_out_of_range_indices():
    q, k, v = sy.make_qkv(1, 1, 8, 4, sy.FP16, 53)
    with pytest.raises(ValueError):
        oracle.attention_bwd_keys(q, k, v, q, sy.FP16, 0.5, True, 1, np.array([0]))
    with pytest.raises(ValueError):
        oracle.attention_bwd_keys(q, k, v, q, sy.FP16, 0.5, True, 0, np.array([8]))
