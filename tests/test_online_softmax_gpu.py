"""The online softmax's moving maximum on the GPU, against the CPU oracle.

The kernels raise a row's running maximum m only when a key tile's maximum
exceeds it by more than 8 in the exp2 domain, and rescale the unnormalised
output O~ by 2^(m_old - m_new) when they do (FlashAttention V2 in depth,
section 3.2, deferred rescaling; Lesson 6.6, "Online softmax").  Random
N(0, 1) workloads almost never trigger that branch, so the inputs here are
built to: key tile t carries a score ramp, so that every tile's maximum
rises past the threshold (the rescale runs on every tile), or stays just
below it (P reaches 2^7.9 without a rescale).  Each construction is checked
on the CPU first, from the 16-bit inputs themselves, so a test cannot pass
on inputs that miss the branch.

Also here: the Flash Attention 2 page's worked example ("Worked Example",
N = 6, d = 2) with its three key tiles placed in three different 64-key
tiles of the GPU kernel, and scales of zero and below (uniform weights;
reversed score order), which the definition S = scale * Q K^T allows.

Tolerances as everywhere: max |O_gpu - O_oracle| <= 2e-3 (fp16), 1e-2
(bf16); max |LSE_gpu - LSE_oracle| <= 1e-3.
"""
import json
import os

import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
import oracle
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu

TOL_O = {sy.FP16: 2e-3, sy.BF16: 1e-2}
TOL_LSE = 1e-3
TORCH_DT = {sy.FP16: torch.float16, sy.BF16: torch.bfloat16}
LOG2E = 1.4426950408889634
KEY_TILE = 64          # keys per tile of the forward kernel at every head dim
THRESHOLD_LOG2 = 8.0   # the running maximum is raised past this margin
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa2_build.build()
    fa2.load_library()
    yield
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "device status word set: 0x%x" % detail


def to_dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(TORCH_DT[dtype])


def status_ok():
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "device status 0x%x" % detail


def check(o, lse, o_ref, lse_ref, dtype, label):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), label + ": non-finite output"
    eo = float(np.abs(o - o_ref).max())
    el = float(np.abs(lse - lse_ref).max())
    print("%s: max|dO| %.3e (tol %.0e)  max|dLSE| %.3e" % (label, eo, TOL_O[dtype], el))
    assert eo <= TOL_O[dtype], "%s: O error %.3e" % (label, eo)
    assert el <= TOL_LSE, "%s: LSE error %.3e" % (label, el)


def run_fwd(q, k, v, dtype, scale, causal):
    o, lse = fa2.fa2_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, causal=causal)
    status_ok()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def bits(x, dtype):
    return sy.f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


def tile_maxima_log2(q, k, dtype, scale, causal):
    """Per (b, h, row): the exp2-domain maximum of the visible scores of each
    64-key tile (NaN where the row sees none of the tile), from the inputs as
    the GPU receives them (16-bit values, widened exactly)."""
    qf, kf = oracle.widen(q, dtype), oracle.widen(k, dtype)
    s = scale * LOG2E * np.einsum("bhid,bhjd->bhij", qf, kf)
    N = q.shape[2]
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    tiles = (N + KEY_TILE - 1) // KEY_TILE
    pad = np.full(s.shape[:3] + (tiles * KEY_TILE - N,), -np.inf)
    m = np.concatenate([s, pad], axis=3).reshape(s.shape[:3] + (tiles, KEY_TILE)).max(axis=4)
    return np.where(np.isneginf(m), np.nan, m)


def ramp_inputs(B, H, N, d, dtype, step, seed, jitter):
    """q_i = e_1 + jitter * r_i e_2 and k_j = step * floor(j / 64) e_1 + jitter * u_j e_2,
    so with scale 1 a score is step * (key tile) plus a small random term.

    The softmax these ramps make is sharp: a row's weight sits on the few keys
    of its last tile, so O comes close to single value rows.  V is uniform in
    [-1, 1], which keeps |O| <= 1, the range in which the tolerances above
    hold for the 16-bit output formats (bf16's half spacing is 2^-9 there; an
    N(0, 1) value row of 4.3 would alone round by up to 2^-6)."""
    rng = np.random.default_rng(seed)
    q = np.zeros((B, H, N, d), np.float32)
    k = np.zeros((B, H, N, d), np.float32)
    q[..., 0] = 1.0
    q[..., 1] = jitter * rng.uniform(-1, 1, size=(B, H, N))
    k[..., 0] = step * (np.arange(N) // KEY_TILE)
    k[..., 1] = jitter * rng.uniform(-1, 1, size=(B, H, N))
    v = rng.uniform(-1, 1, size=(B, H, N, d)).astype(np.float32)
    return bits(q, dtype), bits(k, dtype), bits(v, dtype)


@pytest.mark.parametrize("N", [384, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_rescale_on_every_key_tile(d, dtype, causal, N):
    """Every key tile's maximum exceeds the previous one by more than 8 (exp2
    domain): every row raises its maximum and rescales O~ on every tile it sees."""
    q, k, v = ramp_inputs(1, 2, N, d, dtype, step=10.0, seed=100 + d + N, jitter=0.5)
    m = tile_maxima_log2(q, k, dtype, 1.0, causal)
    jumps = np.diff(m, axis=3)                     # tile t's maximum over tile t-1's
    seen = ~np.isnan(jumps)
    assert seen.sum() > 0 and np.all(jumps[seen] > THRESHOLD_LOG2), "construction misses the rescale branch"
    o, lse = run_fwd(q, k, v, dtype, 1.0, causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, 1.0, causal)
    check(o, lse, o_ref, lse_ref, dtype, "rescale every tile d=%d N=%d causal=%d" % (d, N, causal))


@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_ramp_just_below_rescale_threshold(d, dtype):
    """Tile maxima rise by 7.9 per tile (exp2 domain): tile 1 stays below the
    margin, so its P reaches 2^7.9 on the maximum of tile 0; tile 2 is 15.8
    above it and raises the maximum; tile 3 again stays below."""
    N = 4 * KEY_TILE
    scale = 7.9 / LOG2E
    q, k, v = ramp_inputs(1, 2, N, d, dtype, step=1.0, seed=200 + d, jitter=0.05)
    m = tile_maxima_log2(q, k, dtype, scale, False)
    j01 = m[..., 1] - m[..., 0]
    assert np.all((j01 > 7.5) & (j01 < THRESHOLD_LOG2)), "construction crosses the margin at tile 1"
    assert np.all(m[..., 2] - m[..., 0] > THRESHOLD_LOG2)
    o, lse = run_fwd(q, k, v, dtype, scale, False)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, scale, False)
    check(o, lse, o_ref, lse_ref, dtype, "ramp below the margin d=%d" % d)


def _closed_form(terms):
    return sum(c * np.exp(x) for c, x in terms)


@pytest.mark.parametrize("N", [192, 130])
@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
def test_worked_example_across_three_key_tiles(dtype, N):
    """The page's K tiles 1-3 (keys 1-2, 3-4, 5-6) at key rows 0-1, 64-65 and
    128-129, i.e. in three different tiles of the kernel.  Filler keys score
    -200 for every query (a third column: q = 1, filler k = -200, example keys
    0), so they carry weight exp(-200) ~ 0 and the 6-key example is reproduced
    exactly: row 0 (the page's row 1) sees its maximum move 4 -> 7 -> 10 across
    the kernel's tiles, and rows 0-1 must match the page's numbers."""
    g = json.load(open(os.path.join(GOLDEN, "flash_attention_2_worked_example.json")))
    Q, K, V = np.array(g["Q"], float), np.array(g["K_transposed"], float).T, np.array(g["V"], float)
    d = 64
    q = np.zeros((1, 1, N, d))
    k = np.zeros((1, 1, N, d))
    v = np.zeros((1, 1, N, d))
    q[0, 0, :, 2] = 1.0
    q[0, 0, :6, :2] = Q
    k[0, 0, :, 2] = -200.0
    rows = [0, 1, 64, 65, 128, 129]
    for page_key, r in enumerate(rows):
        k[0, 0, r, :2] = K[page_key]
        k[0, 0, r, 2] = 0.0
        v[0, 0, r, :2] = V[page_key]
    qb, kb, vb = bits(q, dtype), bits(k, dtype), bits(v, dtype)
    # the construction: row 0's visible maxima move across three kernel tiles
    m = tile_maxima_log2(qb, kb, dtype, 1.0, False)[0, 0, 0, :3] / LOG2E
    assert np.allclose(m, [4.0, 7.0, 10.0])
    o, lse = run_fwd(qb, kb, vb, dtype, 1.0, False)
    o_ref, lse_ref = oracle.attention_fwd(qb, kb, vb, dtype, 1.0, False)
    check(o, lse, o_ref, lse_ref, dtype, "worked example across tiles N=%d" % N)
    # the page's own numbers for its rows 1-2: O = O~ / l from the closed forms
    ell = [_closed_form(g["printed_l_final_closed_form"][r]) for r in ("row0", "row1")]
    for i, r in enumerate(("row0", "row1")):
        ot = [_closed_form(t) for t in g["printed_O_tilde_final_closed_form"][r]]
        want = np.array(ot) / ell[i]
        assert np.abs(o[0, 0, i, :2] - want).max() <= TOL_O[dtype]
        assert abs(lse[0, 0, i] - (g["printed_running_max_after_each_step"][2][i] + np.log(ell[i]))) <= TOL_LSE
    assert np.all(o[0, 0, :, 2:] == 0)


# ------------------------------------------------------------------ scale zero and negative

SCALES = {"zero": lambda d: 0.0, "negative": lambda d: -1.0 / np.sqrt(d), "negative x2": lambda d: -2.0 / np.sqrt(d)}


def uniform_values(v_bits, dtype, seed):
    """Value rows uniform in [-1, 1] (|O| <= 1, see ramp_inputs) in place of the N(0, 1) draws."""
    rng = np.random.default_rng(seed)
    return bits(rng.uniform(-1, 1, size=v_bits.shape), dtype)


@pytest.mark.parametrize("which", sorted(SCALES))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_forward_any_finite_scale(d, dtype, causal, which):
    B, H, N = 1, 2, 200
    scale = SCALES[which](d)
    q, k, v = sy.make_qkv(B, H, N, d, dtype, seed=300 + d)
    v = uniform_values(v, dtype, 300 + d)
    o, lse = run_fwd(q, k, v, dtype, scale, causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    check(o, lse, o_ref, lse_ref, dtype, "scale %s d=%d causal=%d" % (which, d, causal))
    if scale == 0.0:
        # uniform weights: O = mean of the visible value rows, L = ln(visible keys)
        n = np.arange(1, N + 1) if causal else np.full(N, N)
        assert np.abs(lse - np.log(n)).max() <= TOL_LSE


@pytest.mark.parametrize("which", ["zero", "negative"])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_general_forward_any_finite_scale(d, which):
    """A band mask (window 40 back, 3 ahead) with N_q != N_k: the element mask
    runs on most tiles, with a zero or negative scale."""
    dtype, nq, nk = sy.BF16, 150, 333
    scale = SCALES[which](d)
    q = sy.make_qkv(1, 2, nq, d, dtype, 400 + d)[0]
    _, k, v = sy.make_qkv(1, 2, nk, d, dtype, 401 + d)
    o, lse = fa2.fa2_fwd_ex(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, window_left=40,
                            window_right=3)
    status_ok()
    o_ref, lse_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_left=40, window_right=3)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, dtype,
          "band scale %s d=%d" % (which, d))


@pytest.mark.parametrize("which", ["zero", "negative"])
@pytest.mark.parametrize("nq", [1, 4])
@pytest.mark.parametrize("d,dtype", [(64, sy.FP16), (128, sy.BF16), (256, sy.FP16)])
def test_decode_any_finite_scale(d, dtype, nq, which):
    nk = 3000
    scale = SCALES[which](d)
    q = sy.make_qkv(2, 2, nq, d, dtype, 500 + d)[0]
    _, k, v = sy.make_qkv(2, 2, nk, d, dtype, 501 + d)
    o, lse = fa2.fa2_decode(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, window_right=0)
    status_ok()
    o_ref, lse_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_right=0)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, dtype,
          "decode scale %s d=%d rows=%d" % (which, d, nq))


BWD_TOL = {sy.FP16: 3e-3, sy.BF16: 1.5e-2}


@pytest.mark.parametrize("which", ["zero", "negative"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,dtype", [(64, sy.FP16), (128, sy.BF16)])
def test_backward_any_finite_scale(d, dtype, causal, which):
    """Gradients relative to their own scale, as in the backward parity tests."""
    B, H, N = 1, 2, 300
    scale = SCALES[which](d)
    q, k, v = sy.make_qkv(B, H, N, d, dtype, 600 + d)
    dout = sy.make_qkv(B, H, N, d, dtype, 601 + d)[0]
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, dout))
    o, lse = fa2.fa2_fwd(tq, tk, tv, scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    status_ok()
    ref = oracle.attention_bwd(q, k, v, dout, dtype, scale, causal)
    common = max(float(np.abs(r).max()) for r in ref[:3])
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3]):
        g = g.double().cpu().numpy()
        assert np.isfinite(g).all(), name
        den = max(float(np.abs(r).max()), 1e-3 * common, 1e-30)
        rel = float(np.abs(g - r).max() / den)
        print("bwd scale %s d=%d %s: %.3e" % (which, d, name, rel))
        assert rel <= BWD_TOL[dtype], "%s: %.3e" % (name, rel)
