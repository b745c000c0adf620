"""Parity of the CUDA forward pass (through the C ABI) with the CPU oracle.

Tolerances: max |O_gpu - O_oracle| <= 2e-3 (fp16) or 1e-2 (bf16), and
max |LSE_gpu - LSE_oracle| <= 1e-3, where the oracle is exact fp64 on the
same 16-bit inputs.  Small sizes are compared element by element over every
output; the full-size workloads are compared on sampled rows (first rows,
tile boundaries, ragged tails, random rows) in the very launch
configuration the benchmark times.
"""
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


def run_gpu(q, k, v, dtype, scale, causal):
    o, lse = fa2.fa2_fwd(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "kernel wait timed out (0x%x)" % detail
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def rounding_floor(o_ref, dtype):
    r = torch.from_numpy(o_ref).to(TORCH_DT[dtype]).double().numpy()
    return float(np.abs(r - o_ref).max()) if o_ref.size else 0.0


def check(o_gpu, lse_gpu, o_ref, lse_ref, dtype, label):
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all(), label + ": non-finite output"
    eo = float(np.abs(o_gpu - o_ref).max())
    el = float(np.abs(lse_gpu - lse_ref).max())
    floor = rounding_floor(o_ref, dtype)
    print("%s: max|dO| %.3e (rounding floor %.3e, tol %.0e)  max|dLSE| %.3e" % (label, eo, floor, TOL_O[dtype], el))
    assert eo <= TOL_O[dtype], "%s: O error %.3e > %.0e (rounding floor %.3e)" % (label, eo, TOL_O[dtype], floor)
    assert el <= TOL_LSE, "%s: LSE error %.3e > %.0e" % (label, el, TOL_LSE)


# ------------------------------------------------------------------ small, every output

SMALL_N = [1, 2, 63, 64, 65, 127, 128, 129, 200, 255, 257, 384]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", SMALL_N)
def test_small_all_outputs(N, d, dtype, causal):
    B, H = (2, 3) if N <= 129 else (1, 2)
    q, k, v = sy.make_qkv(B, H, N, d, dtype, seed=7000 + N + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_gpu(q, k, v, dtype, scale, causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    check(o, lse, o_ref, lse_ref, dtype, "N=%d d=%d %s causal=%d" % (N, d, "bf16" if dtype else "fp16", causal))


@pytest.mark.parametrize("d,dtype,causal", [(128, sy.BF16, True), (64, sy.FP16, False), (256, sy.FP16, True),
                                            (256, sy.BF16, False)])
def test_several_tiles_ragged_all_outputs(d, dtype, causal):
    B, H, N = 1, 2, 1000
    q, k, v = sy.make_qkv(B, H, N, d, dtype, seed=7100 + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_gpu(q, k, v, dtype, scale, causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, scale, causal)
    check(o, lse, o_ref, lse_ref, dtype, "N=1000 d=%d" % d)


# ------------------------------------------------------------------ the pages' examples

def _embed(mat, d):
    """Zero-pad the columns of a small matrix to head dim d (adds 0 to every dot product)."""
    mat = np.asarray(mat, dtype=np.float64)
    out = np.zeros((1, 1, mat.shape[0], d))
    out[0, 0, :, :mat.shape[1]] = mat
    return out


def _bits(x, dtype):
    return sy.f32_to_bits(np.asarray(x, dtype=np.float32), dtype)


@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_worked_example_embedded(dtype, causal):
    Q = [[2, -1], [-2, 5], [4, 1], [0, 2], [3, 0], [1, -3]]
    KT = [[1, 0, 4, -1, 5, 2], [-2, 3, 1, 2, 0, -4]]
    V = [[3, 0], [1, 2], [-2, 1], [5, -3], [4, 0], [-1, 2]]
    q = _bits(_embed(Q, 64), dtype)
    k = _bits(_embed(np.array(KT).T, 64), dtype)
    v = _bits(_embed(V, 64), dtype)
    o, lse = run_gpu(q, k, v, dtype, 1.0, causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, dtype, 1.0, causal)
    check(o, lse, o_ref, lse_ref, dtype, "worked example")
    assert np.all(o[0, 0, :, 2:] == 0)
    if causal:
        assert np.array_equal(o[0, 0, 0, :2], [3.0, 0.0]) and lse[0, 0, 0] == pytest.approx(4.0, abs=1e-5)


def test_practice_row_embedded():
    scores = [1.0, 3.0, 2.0, 5.0, 0.5, 4.0]
    values = [10.0, 20.0, 30.0, 40.0, 50.0, 60.0]
    q = _bits(_embed(np.ones((6, 1)), 64), sy.FP16)
    k = _bits(_embed(np.array(scores).reshape(6, 1), 64), sy.FP16)
    v = _bits(_embed(np.array(values).reshape(6, 1), 64), sy.FP16)
    o, lse = run_gpu(q, k, v, sy.FP16, 1.0, False)
    # |O| = 42.3 is far outside the N(0,1) range the 2e-3 tolerance is set for: fp16 spacing there is
    # 1/32, so the bound is half a spacing for the output rounding plus 2^-11 relative on each P term
    # times its value's distance from O (at most 50): 1/64 + 50 * 2^-11 ~= 0.040
    assert abs(o[0, 0, 0, 0] - 42.347429) <= 1 / 64 + 50 * 2.0 ** -11
    assert lse[0, 0, 0] == pytest.approx(5.0 + np.log(1.5824245), abs=1e-3)


# ------------------------------------------------------------------ full-size workloads

def _sample_rows(w, rng, per_head=48):
    rows = set(range(min(w.N, 8)))
    for b in (127, 128, 129, 255, 256, w.N // 2, w.N - 129, w.N - 128, w.N - 1):
        if 0 <= b < w.N:
            rows.add(b)
    rows.update(range(max(0, w.N - 4), w.N))
    rows.update(int(x) for x in rng.integers(0, w.N, size=per_head))
    return sorted(rows)


@pytest.mark.parametrize("index", [1, 2, 3, 5])
def test_workload_parity_every_output(index):
    """The workload in the benchmark's launch configuration, every element of O
    and LSE against the oracle (which evaluates the whole problem in seconds
    on the host's cores: 1.4e11 - 2.7e11 FLOPs)."""
    w = sy.WORKLOADS[index]
    q, k, v = w.inputs()
    o, lse = run_gpu(q, k, v, w.dtype, w.scale, w.causal)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, w.dtype, w.scale, w.causal)
    check(o, lse, o_ref, lse_ref, w.dtype, w.name + " (every output)")


def test_workload_parity_every_head_sampled_rows():
    """The long-context workload (B1 H32 N16384 d128 causal, 2.2e12 FLOPs: too
    much for the oracle whole) on sampled rows of every head -- tile
    boundaries, the first and last rows and random rows -- so that a tile
    written into the wrong head or position shows up in some head; plus
    properties that hold for every output."""
    w = sy.WORKLOADS[4]
    q, k, v = w.inputs()
    o, lse = run_gpu(q, k, v, w.dtype, w.scale, w.causal)
    BH = w.B * w.H
    rng = np.random.default_rng(4)
    bh_idx, row_idx = [], []
    for bh in range(BH):
        rows = _sample_rows(w, rng, per_head=24)
        bh_idx += [bh] * len(rows)
        row_idx += rows
    bh_idx = np.array(bh_idx)
    row_idx = np.array(row_idx)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.dtype, w.scale, w.causal, bh_idx, row_idx)
    o_flat = o.reshape(BH, w.N, w.d)[bh_idx, row_idx]
    lse_flat = lse.reshape(BH, w.N)[bh_idx, row_idx]
    check(o_flat, lse_flat, o_ref, lse_ref, w.dtype, w.name + " (%d sampled rows, every head)" % len(row_idx))
    # properties that hold at any size, checked on every output
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vmax = np.abs(sy.bits_to_f32(v, w.dtype)).max()
    assert np.abs(o).max() <= vmax * (1 + 1e-2)      # a convex combination of value rows
    # causal row 0 of every head sees only key 0: O = V_0 (rounded once) and L = scale q_0 . k_0
    v0 = sy.bits_to_f32(v, w.dtype).reshape(BH, w.N, w.d)[:, 0]
    assert np.array_equal(o.reshape(BH, w.N, w.d)[:, 0], v0.astype(np.float64))


# ------------------------------------------------------------------ behaviour

def test_deterministic():
    w = sy.Workload(0, 1, 4, 777, 128, sy.BF16, True)
    q, k, v = w.inputs()
    a = run_gpu(q, k, v, w.dtype, w.scale, True)
    b = run_gpu(q, k, v, w.dtype, w.scale, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_outputs_written_in_place_only():
    # o and lse live inside larger buffers filled with a canary; nothing outside may change
    B, H, N, d = 1, 2, 300, 128
    q, k, v = sy.make_qkv(B, H, N, d, sy.FP16, 77)
    pad = 8192
    o_buf = torch.full((pad * 2 + B * H * N * d,), 12345.0, dtype=torch.float16, device="cuda")
    l_buf = torch.full((pad * 2 + B * H * N,), -777.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * H * N * d].view(B, H, N, d)
    lse = l_buf[pad:pad + B * H * N].view(B, H, N)
    fa2.fa2_fwd(to_dev(q, sy.FP16), to_dev(k, sy.FP16), to_dev(v, sy.FP16), o, lse, causal=True)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 12345.0) and torch.all(o_buf[pad + B * H * N * d:] == 12345.0)
    assert torch.all(l_buf[:pad] == -777.0) and torch.all(l_buf[pad + B * H * N:] == -777.0)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, sy.FP16, 1 / np.sqrt(d), True)
    check(o.double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref, sy.FP16, "in-place")


def test_side_stream_and_host_entry_point():
    # small problem: the host path runs copy-in, forward and copy-out in one pass
    B, H, N, d = 2, 2, 333, 64
    q, k, v = sy.make_qkv(B, H, N, d, sy.BF16, 78)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o_d, l_d = fa2.fa2_fwd(to_dev(q, sy.BF16), to_dev(k, sy.BF16), to_dev(v, sy.BF16), stream=s)
    s.synchronize()
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (q, k, v))
    oh = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa2.fa2_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa2.fa2_fwd_host(qh, kh, vh, oh, lh, ws)
    assert torch.equal(oh, o_d.cpu()) and torch.equal(lh, l_d.cpu())


def test_invalid_device_arguments_launch_nothing():
    x = torch.zeros(1 * 1 * 64 * 64 + 8, dtype=torch.float16, device="cuda")
    lse = torch.zeros(64 + 4, dtype=torch.float32, device="cuda")
    lib = fa2.load_library()
    base = x.data_ptr()
    rc = lib.fa2_fwd(base + 2, base, base, base, lse.data_ptr(), 1, 1, 64, 64, 0.125, 0, 0, None)
    assert rc == fa2.FA2_ERR_MISALIGNED
    rc = lib.fa2_fwd(base, base, base, base, lse.data_ptr(), 1, 1, 64, 64, 0.125, 0, 0, None)
    assert rc == fa2.FA2_ERR_INVALID_ARG           # o aliases q
    torch.cuda.synchronize()


@pytest.mark.parametrize("d,dtype,causal,N", [(256, sy.FP16, False, 3000), (256, sy.BF16, True, 1000),
                                              (128, sy.BF16, True, 2048), (64, sy.FP16, False, 1024)])
def test_repeated_launches_identical(d, dtype, causal, N):
    """Many back-to-back launches: every one bit-identical and no wait ever timing out.

    Pipeline races (a barrier running a phase ahead of its waiter) show up as
    rare timeouts or wrong tiles under varying timing, not on a single run."""
    B, H = 1, 16
    q, k, v = (to_dev(x, dtype) for x in sy.make_qkv(B, H, N, d, dtype, seed=7200 + d + N))
    o0, l0 = fa2.fa2_fwd(q, k, v, causal=causal)
    o, lse = torch.empty_like(o0), torch.empty_like(l0)
    for i in range(60):
        fa2.fa2_fwd(q, k, v, o, lse, causal=causal)
        if i % 10 == 9:
            torch.cuda.synchronize()
            assert torch.equal(o, o0) and torch.equal(lse, l0), "launch %d differs" % i
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "a wait timed out (0x%x)" % detail


def test_host_entry_point_pipelined_over_head_groups():
    # >= 48 MB of input: the host path overlaps copies of one group of heads with the forward of another
    B, H, N, d = 1, 16, 8192, 64
    q, k, v = sy.make_qkv(B, H, N, d, sy.FP16, 79)
    o_d, l_d = fa2.fa2_fwd(to_dev(q, sy.FP16), to_dev(k, sy.FP16), to_dev(v, sy.FP16), causal=True)
    torch.cuda.synchronize()
    qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.float16).pin_memory() for x in (q, k, v))
    oh = torch.empty((B, H, N, d), dtype=torch.float16).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa2.fa2_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        oh.zero_()
        lh.zero_()
        fa2.fa2_fwd_host(qh, kh, vh, oh, lh, ws, causal=True)
        assert torch.equal(oh, o_d.cpu()) and torch.equal(lh, l_d.cpu())
