"""Pins for the CPU oracle: values the pages print, closed forms, invariants and
a high-precision brute force -- each chosen so a plausible slip in the oracle
(dropped term, wrong sign or index, transposed operand, wrong mask side,
wrong log base) fails at least one of them.  CPU only."""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

import oracle
from oracle.tiled_reference import tiled_attention
from exact_tiled_attention_fa2_gb300 import synthetic as sy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _fp16_bits(x):
    a = np.asarray(x, dtype=np.float64)
    b = a.astype(np.float16)
    assert np.array_equal(b.astype(np.float64), a), "fixture values must be exact in fp16"
    return b.view(np.uint16)


def _closed(terms):
    return sum(c * math.exp(x) for c, x in terms)


def _as4(a):
    a = np.asarray(a)
    return a.reshape((1, 1) + a.shape)


# ---------------------------------------------------------------- worked example

def _worked():
    g = _load("flash_attention_2_worked_example.json")
    Q = np.array(g["Q"], dtype=np.float64)
    K = np.array(g["K_transposed"], dtype=np.float64).T
    V = np.array(g["V"], dtype=np.float64)
    return g, Q, K, V


def test_worked_example_closed_forms():
    g, Q, K, V = _worked()
    o, lse = oracle.attention_fwd(_as4(_fp16_bits(Q)), _as4(_fp16_bits(K)), _as4(_fp16_bits(V)),
                                  oracle.FP16, g["scale"], False)
    o, lse = o[0, 0], lse[0, 0]
    lcf = g["printed_l_final_closed_form"]
    ocf = g["printed_O_tilde_final_closed_form"]
    m_final = g["printed_running_max_after_each_step"][-1]
    for r, key in enumerate(["row0", "row1"]):
        l_r = _closed(lcf[key])
        for c in range(2):
            assert o[r, c] == pytest.approx(_closed(ocf[key][c]) / l_r, abs=1e-12)
        # L = m + ln(l): natural log, in the (unscaled here) score domain
        assert lse[r] == pytest.approx(m_final[r] + math.log(l_r), abs=1e-12)


def test_worked_example_printed_values():
    g, Q, K, V = _worked()
    o, _ = oracle.attention_fwd(_as4(_fp16_bits(Q)), _as4(_fp16_bits(K)), _as4(_fp16_bits(V)),
                                oracle.FP16, 1.0, False)
    o = o[0, 0]
    half = 0.5 * 10 ** -g["printed_decimals"]
    printed = np.array(g["printed_O_final_approx"])
    for r in range(2):
        for c in range(2):
            if (r, c) == (0, 0):
                # the page's printed 3.173 is a slip (its closed form gives 3.176591)
                assert abs(o[r, c] - printed[r, c]) > 2 * half
                continue
            assert abs(o[r, c] - printed[r, c]) <= half + 1e-12


def test_worked_example_tiled_trace_matches_page():
    g, Q, K, V = _worked()
    trace = []
    O, L = tiled_attention(Q, K, V, B_r=2, B_c=2, scale=1.0, trace=trace)
    steps = [t for t in trace if t["i"] == 0]
    assert len(steps) == 3
    for t, s_print, m_print in zip(steps, g["printed_S_tiles_for_Q1"], g["printed_running_max_after_each_step"]):
        np.testing.assert_array_equal(t["S"], np.array(s_print, dtype=np.float64))
        np.testing.assert_array_equal(t["m"], np.array(m_print, dtype=np.float64))
    last = steps[-1]
    lcf = g["printed_l_final_closed_form"]
    ocf = g["printed_O_tilde_final_closed_form"]
    for r, key in enumerate(["row0", "row1"]):
        assert last["l"][r] == pytest.approx(_closed(lcf[key]), abs=1e-12)
        assert last["l"][r] == pytest.approx(g["printed_l_final_approx"][r], abs=0.5e-4)
        for c in range(2):
            assert last["O_tilde"][r, c] == pytest.approx(_closed(ocf[key][c]), abs=1e-12)
    full, _ = oracle.attention_fwd(_as4(_fp16_bits(Q)), _as4(_fp16_bits(K)), _as4(_fp16_bits(V)),
                                   oracle.FP16, 1.0, False)
    np.testing.assert_allclose(O, full[0, 0], atol=1e-12, rtol=0)


def test_worked_example_causal_row0():
    g, Q, K, V = _worked()
    o, lse = oracle.attention_fwd(_as4(_fp16_bits(Q)), _as4(_fp16_bits(K)), _as4(_fp16_bits(V)),
                                  oracle.FP16, 1.0, True)
    np.testing.assert_array_equal(o[0, 0, 0], V[0])          # only key 0 is visible: O_0 = V_0
    assert lse[0, 0, 0] == pytest.approx(Q[0] @ K[0], abs=0)  # L_0 = s_00 = 4
    assert lse[0, 0, 0] == 4.0


# ---------------------------------------------------------------- practice row

def test_practice_row_online_equals_direct():
    g = _load("lesson_6_6_practice_row.json")
    s = np.array(g["scores"])
    v = np.array(g["values"])
    n = len(s)
    # embed: q = [1], k_j = [s_j], v_j = [value_j], scale 1  ->  s_ij = s_j
    q = _fp16_bits(np.ones((1, 1, n, 1)))
    k = _fp16_bits(s.reshape(1, 1, n, 1))
    vv = _fp16_bits(v.reshape(1, 1, n, 1))
    o, lse = oracle.attention_fwd(q, k, vv, oracle.FP16, 1.0, False)
    assert abs(o[0, 0, 0, 0] - g["printed_online"]) <= 0.5e-6
    assert abs(o[0, 0, 0, 0] - g["printed_direct"]) <= 0.5e-6
    # L = max + ln(l_final): the printed final l carries 4 decimals
    l_print = g["printed_blocks"][-1]["l"]
    assert abs(lse[0, 0, 0] - (5.0 + math.log(l_print))) <= 0.5e-4 / l_print + 1e-12


def test_practice_row_block_trace_and_block_size_invariance():
    g = _load("lesson_6_6_practice_row.json")
    s = np.array(g["scores"]).reshape(1, -1)
    v = np.array(g["values"]).reshape(-1, 1)
    Q = np.ones((1, 1))
    K = s.reshape(-1, 1)
    trace = []
    O, _ = tiled_attention(Q, K, v, B_r=1, B_c=g["block"], trace=trace)
    dec = g["printed_decimals"]
    m_prev = -math.inf
    for t, p in zip(trace, g["printed_blocks"]):
        m = t["m"][0]
        assert abs(m - p["m"]) <= 0.5 * 10 ** -dec["m"]
        scale = math.exp(m_prev - m)
        assert abs(scale - p["scale"]) <= 0.5 * 10 ** -dec["scale"]
        assert abs(t["l"][0] - p["l"]) <= 0.5 * 10 ** -dec["l"]
        assert abs(t["O_tilde"][0, 0] / t["l"][0] - p["output_so_far"]) <= 0.5 * 10 ** -dec["output_so_far"]
        m_prev = m
    # "Set BLOCK = 1, then BLOCK = 3": the final answer does not move
    for block in (1, 2, 3, 6):
        Ob, _ = tiled_attention(Q, K, v, B_r=1, B_c=block)
        assert abs(Ob[0, 0] - g["printed_online"]) <= 0.5e-6


# ---------------------------------------------------------------- invariants

def _rand_bits(shape, dtype, seed):
    B, H, N, d = shape
    return sy.make_qkv(B, H, N, d, dtype, seed)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
def test_softmax_rows_sum_to_one(dtype):
    # V = identity (d = N) makes O equal to P itself
    N = 12
    q, k, _ = _rand_bits((1, 2, N, N), dtype, 11)
    eye = np.broadcast_to(np.eye(N), (1, 2, N, N))
    v = sy.f32_to_bits(eye.astype(np.float32), dtype).reshape(1, 2, N, N)
    for causal in (False, True):
        o, _ = oracle.attention_fwd(q, k, v, dtype, 0.3, causal)
        np.testing.assert_allclose(o.sum(axis=-1), 1.0, atol=1e-12, rtol=0)
        assert (o >= 0).all()
        if causal:
            assert np.all(o[..., np.triu_indices(N, 1)[0], np.triu_indices(N, 1)[1]] == 0)


def test_identical_keys_give_mean_of_values():
    B, H, N, d = 1, 3, 9, 5
    q, k, v = _rand_bits((B, H, N, d), oracle.BF16, 12)
    k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    scale = 0.7
    o, lse = oracle.attention_fwd(q, k, v, oracle.BF16, scale, False)
    Vd = oracle.widen(v, oracle.BF16)
    Qd = oracle.widen(q, oracle.BF16)
    Kd = oracle.widen(k, oracle.BF16)
    np.testing.assert_allclose(o, np.broadcast_to(Vd.mean(axis=2, keepdims=True), o.shape), atol=1e-12, rtol=0)
    s = scale * np.einsum("bhnd,bhd->bhn", Qd, Kd[:, :, 0, :])
    np.testing.assert_allclose(lse, s + math.log(N), atol=1e-12, rtol=0)


def test_single_key():
    q, k, v = _rand_bits((2, 2, 1, 7), oracle.FP16, 13)
    o, lse = oracle.attention_fwd(q, k, v, oracle.FP16, 0.25, False)
    Vd, Qd, Kd = (oracle.widen(x, oracle.FP16) for x in (v, q, k))
    np.testing.assert_array_equal(o, Vd)
    np.testing.assert_allclose(lse, 0.25 * (Qd * Kd).sum(-1), atol=1e-13, rtol=0)


def test_constant_value_rows():
    B, H, N, d = 1, 2, 17, 4
    q, k, v = _rand_bits((B, H, N, d), oracle.FP16, 14)
    v = np.broadcast_to(v[:, :, 3:4, :], v.shape).copy()
    for causal in (False, True):
        o, _ = oracle.attention_fwd(q, k, v, oracle.FP16, 0.5, causal)
        np.testing.assert_allclose(o, oracle.widen(v, oracle.FP16), atol=1e-13, rtol=0)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
def test_causal_row0_and_prefix_rule(dtype):
    mask = np.array(_load("causal_mask_n4.json")["visible"], dtype=bool)
    B, H, N, d = 1, 2, 4, 3
    q, k, v = _rand_bits((B, H, N, d), dtype, 15)
    scale = 0.9
    o, lse = oracle.attention_fwd(q, k, v, dtype, scale, True)
    Qd, Kd, Vd = (oracle.widen(x, dtype) for x in (q, k, v))
    np.testing.assert_array_equal(o[:, :, 0], Vd[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * (Qd[:, :, 0] * Kd[:, :, 0]).sum(-1), atol=1e-13, rtol=0)
    for i in range(N):
        # the printed mask's visible keys for row i are exactly the prefix 0..i, so causal row i
        # equals the last row of the unmasked problem on that prefix
        keys = np.nonzero(mask[i])[0]
        np.testing.assert_array_equal(keys, np.arange(i + 1))
        sub_o, sub_l = oracle.attention_fwd(q[:, :, :i + 1].copy(), k[:, :, keys].copy(), v[:, :, keys].copy(),
                                            dtype, scale, False)
        np.testing.assert_allclose(o[:, :, i], sub_o[:, :, i], atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[:, :, i], sub_l[:, :, i], atol=1e-14, rtol=0)


def test_key_permutation_invariance():
    q, k, v = _rand_bits((1, 2, 23, 6), oracle.BF16, 16)
    perm = np.random.default_rng(0).permutation(23)
    o1, l1 = oracle.attention_fwd(q, k, v, oracle.BF16, 0.4, False)
    o2, l2 = oracle.attention_fwd(q, k[:, :, perm].copy(), v[:, :, perm].copy(), oracle.BF16, 0.4, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-13, rtol=0)
    # permuting V alone (keys fixed) must change the answer: V is indexed by key
    o3, _ = oracle.attention_fwd(q, k, v[:, :, perm].copy(), oracle.BF16, 0.4, False)
    assert np.abs(o3 - o1).max() > 1e-3


def test_scale_multiplies_scores():
    q, k, v = _rand_bits((1, 1, 10, 8), oracle.FP16, 17)
    q2 = sy.f32_to_bits(2.0 * sy.bits_to_f32(q, oracle.FP16), oracle.FP16)   # exact doubling
    o1, l1 = oracle.attention_fwd(q, k, v, oracle.FP16, 0.6, False)
    o2, l2 = oracle.attention_fwd(q2, k, v, oracle.FP16, 0.3, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(l1, l2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_gives_uniform_weights(causal):
    # S = 0 * Q K^T: every visible key has the same weight, so O is the mean of
    # the visible value rows and L = ln(number of visible keys) (closed form)
    N, d = 13, 8
    q, k, v = _rand_bits((2, 1, N, d), oracle.BF16, 21)
    o, lse = oracle.attention_fwd(q, k, v, oracle.BF16, 0.0, causal)
    vf = sy.bits_to_f32(v, oracle.BF16).astype(np.float64)
    for i in range(N):
        n = i + 1 if causal else N
        np.testing.assert_allclose(o[:, :, i], vf[:, :, :n].mean(axis=2), atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=1e-13, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale_equals_negated_queries(causal):
    # scale * (q . k) with scale < 0 equals |scale| * ((-q) . k); negating a
    # 16-bit value flips its sign bit, so both problems are computed exactly alike
    q, k, v = _rand_bits((1, 2, 11, 8), oracle.FP16, 23)
    q_neg = q ^ np.uint16(0x8000)
    o1, l1 = oracle.attention_fwd(q, k, v, oracle.FP16, -0.7, causal)
    o2, l2 = oracle.attention_fwd(q_neg, k, v, oracle.FP16, 0.7, causal)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and the order of the weights reverses: the smallest score gets the largest weight
    o3, _ = oracle.attention_fwd(q, k, v, oracle.FP16, 0.7, causal)
    assert not np.allclose(o1, o3)


def test_very_negative_scores_stay_finite():
    # every score near -2000: exp without the max shift underflows to 0/0
    N, d = 5, 2
    q = np.zeros((1, 1, N, d)); q[..., 0] = -40.0
    k = np.zeros((1, 1, N, d)); k[..., 0] = 50.0 + np.arange(N)
    v = np.arange(N * d, dtype=np.float64).reshape(1, 1, N, d)
    o, lse = oracle.attention_fwd(_fp16_bits(q), _fp16_bits(k), _fp16_bits(v), oracle.FP16, 1.0, False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    s = -40.0 * (50.0 + np.arange(N))
    w = np.exp(s - s.max()); w /= w.sum()
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(w @ v[0, 0], (N, d)), atol=1e-12, rtol=0)


def _brute(Qd, Kd, Vd, scale, causal):
    getcontext().prec = 50
    N, d = Qd.shape
    O = np.zeros((N, d))
    L = np.zeros(N)
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        ex = []
        for j in keys:
            s = Decimal(repr(scale)) * sum(Decimal(repr(float(Qd[i, c]))) * Decimal(repr(float(Kd[j, c])))
                                           for c in range(d))
            ex.append((j, s.exp()))               # no max shift: direct sum of exponentials
        tot = sum(e for _, e in ex)
        for c in range(d):
            O[i, c] = float(sum(e * Decimal(repr(float(Vd[j, c]))) for j, e in ex) / tot)
        L[i] = float(tot.ln())
    return O, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
def test_brute_force_tiny(causal, dtype):
    B, H, N, d = 1, 2, 5, 3
    q, k, v = _rand_bits((B, H, N, d), dtype, 18 + dtype)
    o, lse = oracle.attention_fwd(q, k, v, dtype, 0.8, causal)
    for h in range(H):
        Qd, Kd, Vd = (oracle.widen(x[0, h], dtype) for x in (q, k, v))
        Ob, Lb = _brute(Qd, Kd, Vd, 0.8, causal)
        np.testing.assert_allclose(o[0, h], Ob, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse[0, h], Lb, atol=1e-13, rtol=0)


def test_rows_api_matches_full_api():
    q, k, v = _rand_bits((2, 3, 37, 16), oracle.BF16, 20)
    o, lse = oracle.attention_fwd(q, k, v, oracle.BF16, 0.25, True)
    bh = np.array([0, 0, 4, 4, 5, 2])
    rows = np.array([0, 36, 5, 17, 30, 1])
    o_r, l_r = oracle.attention_rows(q, k, v, oracle.BF16, 0.25, True, bh, rows)
    for t in range(len(bh)):
        b, h = divmod(int(bh[t]), 3)
        np.testing.assert_array_equal(o_r[t], o[b, h, rows[t]])
        assert l_r[t] == lse[b, h, rows[t]]


def test_widening_matches_library_conversions():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    h = allbits.view(np.float16)
    ok = np.isfinite(h)
    np.testing.assert_array_equal(oracle.widen(allbits, oracle.FP16)[ok], h[ok].astype(np.float64))
    assert np.isnan(oracle.widen(allbits, oracle.FP16)[np.isnan(h)]).all()
    f = (allbits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    ok = np.isfinite(f)
    np.testing.assert_array_equal(oracle.widen(allbits, oracle.BF16)[ok], f[ok].astype(np.float64))


def test_invalid_arguments_rejected():
    q, k, v = _rand_bits((1, 1, 4, 2), oracle.FP16, 21)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, 7, 1.0, False)
    with pytest.raises(ValueError):
        oracle.attention_fwd(q, k, v, oracle.FP16, float("nan"), False)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, k, v, oracle.FP16, 1.0, False, [0], [4])


# ---------------------------------------------------------------- tiling is exact

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B_r,B_c", [(1, 1), (2, 2), (3, 2), (2, 3), (64, 64), (16, 5)])
def test_tiled_algorithm_equals_definition(causal, B_r, B_c):
    N, d = 70, 8
    q, k, v = _rand_bits((1, 1, N, d), oracle.BF16, 22)
    o, lse = oracle.attention_fwd(q, k, v, oracle.BF16, 0.35, causal)
    Qd, Kd, Vd = (oracle.widen(x[0, 0], oracle.BF16) for x in (q, k, v))
    for kw in ({}, {"local_max": True}, {"fa1_update": True}):
        O, L = tiled_attention(Qd, Kd, Vd, B_r, B_c, scale=0.35, causal=causal, **kw)
        np.testing.assert_allclose(O, o[0, 0], atol=1e-12, rtol=0)
        np.testing.assert_allclose(L, lse[0, 0], atol=1e-12, rtol=0)


def test_three_named_slips_each_break_exactness():
    N, d = 40, 4
    q, k, v = _rand_bits((1, 1, N, d), oracle.FP16, 23)
    Qd, Kd, Vd = (oracle.widen(x[0, 0], oracle.FP16) for x in (q, k, v))
    o, _ = oracle.attention_fwd(q, k, v, oracle.FP16, 1.0, False)
    ok, _ = tiled_attention(Qd, Kd, Vd, 8, 8)
    assert np.abs(ok - o[0, 0]).max() < 1e-12
    bad, _ = tiled_attention(Qd, Kd, Vd, 8, 8, rescale_output=False)      # l rescaled, O not
    assert np.abs(bad - o[0, 0]).max() > 1e-3
    bad, _ = tiled_attention(Qd, Kd, Vd, 8, 8, normalize_in_loop=True)    # divide inside the loop
    assert np.abs(bad - o[0, 0]).max() > 1e-3
    # m starting at 0: every score very negative -> the shift never happens and exp underflows
    qn = -60.0 * np.abs(Qd)
    kn = 60.0 * np.abs(Kd)
    good, _ = tiled_attention(qn, kn, Vd, 8, 8)
    bad, _ = tiled_attention(qn, kn, Vd, 8, 8, m_init=0.0)
    assert np.isfinite(good).all()
    assert not np.isfinite(bad).all() or np.abs(bad - good).max() > 1e-3


def test_workload_flop_counts():
    w = sy.WORKLOADS[4]
    assert w.flops() == 4.0 * 1 * 32 * 16384 ** 2 * 128 / 2
    assert sy.WORKLOADS[2].flops() == 4.0 * 8 * 16 * 2048 ** 2 * 64
    assert sy.WORKLOADS[1].algorithmic_bytes() == 66048
