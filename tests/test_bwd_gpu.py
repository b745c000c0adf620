"""Parity of the backward pass (fa2_bwd, through the C ABI) with the CPU oracle.

The gradients are compared relative to their own scale: max|g - g_oracle| <=
TOL * max|g_oracle| per tensor.  The pages fix no backward tolerance; TOL is
derived from the arithmetic: P and dS are rounded to the input type before
the products (2^-9 relative in bf16, 2^-12 in fp16), O is read back 16-bit
for D = rowsum(dO o O), and the outputs are rounded once more; the
accumulations over keys and queries add these errors with random signs.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
import oracle
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu

# measured on GB300: <= 6.5e-4 (fp16) and <= 4.6e-3 (bf16) of the gradient scale
TOL = {sy.FP16: 3e-3, sy.BF16: 1.5e-2}
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


def run_bwd(B, H, N, d, dtype, causal, seed):
    q, k, v = sy.make_qkv(B, H, N, d, dtype, seed)
    dout = sy.make_qkv(B, H, N, d, dtype, seed + 500)[0]
    scale = 1.0 / np.sqrt(d)
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, dout))
    o, lse = fa2.fa2_fwd(tq, tk, tv, scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "kernel wait timed out (0x%x)" % detail
    ref = oracle.attention_bwd(q, k, v, dout, dtype, scale, causal)
    return [g.double().cpu().numpy() for g in (dq, dk, dv)], ref


def check(got, ref, dtype, label):
    worst = 0.0
    # each gradient against its own scale, floored at 1e-3 of the largest one's
    # (a gradient can be exactly zero, e.g. dQ and dK when there is a single key)
    common = max(float(np.abs(r).max()) for r in ref[:3])
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref[:3]):
        assert np.isfinite(g).all(), "%s %s: non-finite" % (label, name)
        den = max(float(np.abs(r).max()), 1e-3 * common, 1e-30)
        rel = float(np.abs(g - r).max() / den)
        print("%s %s: max|err|/max|ref| = %.3e (max|ref| %.3e)" % (label, name, rel, den))
        worst = max(worst, rel)
        assert rel <= TOL[dtype], "%s %s: %.3e > %.0e" % (label, name, rel, TOL[dtype])
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [sy.FP16, sy.BF16])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 63, 128, 129, 300])
def test_bwd_small(N, d, dtype, causal):
    B, H = (2, 2) if N <= 129 else (1, 2)
    got, ref = run_bwd(B, H, N, d, dtype, causal, 9000 + N + d)
    check(got, ref, dtype, "N=%d d=%d %s causal=%d" % (N, d, "bf16" if dtype else "fp16", causal))


@pytest.mark.parametrize("d,dtype,causal", [(128, sy.BF16, True), (64, sy.FP16, False), (256, sy.FP16, False),
                                            (256, sy.BF16, True)])
def test_bwd_several_tiles(d, dtype, causal):
    got, ref = run_bwd(1, 2, 1000, d, dtype, causal, 9100 + d)
    check(got, ref, dtype, "N=1000 d=%d" % d)


def test_bwd_rejects_unsupported_head_dim():
    q = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa2.Fa2Error) as e:
        fa2.fa2_bwd(q, q.clone(), q.clone(), q.clone(), torch.zeros(1, 1, 64, device="cuda"), q.clone())
    assert e.value.code == fa2.FA2_ERR_UNSUPPORTED


@pytest.mark.parametrize("index", [2, 3, 5])
def test_bwd_workload_heads(index):
    """The full workload's backward in the benchmark's launch configuration;
    two whole heads (first and last) checked against the oracle."""
    w = sy.WORKLOADS[index]
    q, k, v = w.inputs()
    dout = sy.make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed(0) + 500)[0]
    tq, tk, tv, tdo = (to_dev(x, w.dtype) for x in (q, k, v, dout))
    o, lse = fa2.fa2_fwd(tq, tk, tv, scale=w.scale, causal=w.causal)
    dq, dk, dv = fa2.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    assert fa2.fa2_get_device_status()[0] == fa2.FA2_OK
    got_all = [g.double().cpu().numpy() for g in (dq, dk, dv)]
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        sl = lambda x: np.ascontiguousarray(x[b:b + 1, h:h + 1])
        ref = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(dout), w.dtype, w.scale, w.causal)
        check([g[b:b + 1, h:h + 1] for g in got_all], ref, w.dtype, "%s head (%d,%d)" % (w.name, b, h))
