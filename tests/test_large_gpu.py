"""The forward and backward passes on tensors past 2^31 elements (4 GiB each),
against the oracle.

Element offsets of the last heads' rows exceed 32 bits there, and the row
coordinates reach 262143, so any 32-bit product in the index arithmetic of the
kernels or the host (tensor maps, the LSE and O row offsets, the grid) shows
up as a wrong or missing row.  The inputs are drawn on the device from a seeded
generator (N(0, 1) in fp32, rounded once to the 16-bit type), one head at a
time; the oracle recomputes sampled rows of the first and the last heads from
those heads' own inputs copied back to the host.  The backward is checked on
sampled dQ rows and, under the causal mask, on the dK and dV rows of the last
keys (which only the last query rows see, so the oracle's keys pass stays
small).

Tolerances as in test_parity_gpu: max |O - O_oracle| <= 2e-3 (fp16) or 1e-2
(bf16) and max |LSE - LSE_oracle| <= 1e-3; for the gradients, as in
test_bwd_gpu: max |g - g_oracle| <= TOL * max |g_oracle| over the sampled
rows, TOL = 3e-3 (fp16) or 1.5e-2 (bf16).
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
TOL_GRAD = {sy.FP16: 3e-3, sy.BF16: 1.5e-2}
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


def device_inputs(B, H, N, d, dtype, seed):
    """q, k, v [B, H, N, d] of the 16-bit type, drawn head by head on the device."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = []
    for _ in range(3):
        t = torch.empty((B, H, N, d), dtype=TORCH_DT[dtype], device="cuda")
        for b in range(B):
            for h in range(H):
                t[b, h] = torch.randn((N, d), generator=g, device="cuda", dtype=torch.float32).to(TORCH_DT[dtype])
        out.append(t)
    return out


def head_bits(t, b, h):
    return t[b, h].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)[None, None]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (1, 64, 262144, 128, sy.BF16, True),
    (1, 256, 131072, 64, sy.FP16, False),
    (1, 32, 262144, 256, sy.FP16, True),
])
def test_tensors_past_two_to_the_31_elements(B, H, N, d, dtype, causal):
    assert B * H * N * d >= 1 << 31
    q, k, v = device_inputs(B, H, N, d, dtype, seed=9000 + d)
    scale = d ** -0.5
    o, lse = fa2.fa2_fwd(q, k, v, scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "kernel wait timed out (0x%x)" % detail
    rng = np.random.default_rng(d)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 129, N - 128, N - 1],
                                     rng.integers(0, N, size=8)]))
    for b, h in ((0, 0), (B - 1, H - 1)):
        qb, kb, vb = head_bits(q, b, h), head_bits(k, b, h), head_bits(v, b, h)
        o_ref, lse_ref = oracle.attention_rows(qb, kb, vb, dtype, scale, causal,
                                               np.zeros(rows.size, np.int64), rows)
        o_gpu = o[b, h, torch.from_numpy(rows).cuda()].double().cpu().numpy()
        lse_gpu = lse[b, h, torch.from_numpy(rows).cuda()].double().cpu().numpy()
        assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all()
        eo = float(np.abs(o_gpu - o_ref).max())
        el = float(np.abs(lse_gpu - lse_ref).max())
        print("B%d H%d N%d d%d head (%d, %d): max|dO| %.3e  max|dLSE| %.3e" % (B, H, N, d, b, h, eo, el))
        assert eo <= TOL_O[dtype], "head (%d, %d): O error %.3e" % (b, h, eo)
        assert el <= TOL_LSE, "head (%d, %d): LSE error %.3e" % (b, h, el)
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def device_tensor(B, H, N, d, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    t = torch.empty((B, H, N, d), dtype=TORCH_DT[dtype], device="cuda")
    for b in range(B):
        for h in range(H):
            t[b, h] = torch.randn((N, d), generator=g, device="cuda", dtype=torch.float32).to(TORCH_DT[dtype])
    return t


def grad_check(got, ref, dtype, label, common):
    assert np.isfinite(got).all(), label + ": non-finite"
    den = max(float(np.abs(ref).max()), 1e-3 * common, 1e-30)
    rel = float(np.abs(got - ref).max() / den)
    print("%s: max|err|/den = %.3e (den %.3e, own max|ref| %.3e)" % (label, rel, den, float(np.abs(ref).max())))
    assert rel <= TOL_GRAD[dtype], "%s: %.3e > %.0e" % (label, rel, TOL_GRAD[dtype])


@pytest.mark.parametrize("B,H,N,d,dtype", [
    (1, 64, 262144, 128, sy.BF16),
    (1, 128, 262144, 64, sy.FP16),
    (1, 32, 262144, 256, sy.FP16),
])
def test_backward_past_two_to_the_31_elements(B, H, N, d, dtype):
    assert B * H * N * d >= 1 << 31
    causal = True
    q, k, v = device_inputs(B, H, N, d, dtype, seed=9500 + d)
    dout = device_tensor(B, H, N, d, dtype, seed=9600 + d)
    scale = d ** -0.5
    o, lse = fa2.fa2_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(q, k, v, o, lse, dout, scale=scale, causal=causal)
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "kernel wait timed out (0x%x)" % detail
    del o, lse
    rng = np.random.default_rng(d + 1)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 129, N - 1], rng.integers(0, N, size=6)]))
    keys = np.unique(np.concatenate([[N - 64, N - 63, N - 2, N - 1], rng.integers(N - 64, N, size=4)]))
    for b, h in ((0, 0), (B - 1, H - 1)):
        qb, kb, vb, dob = (head_bits(t, b, h) for t in (q, k, v, dout))
        dq_ref, _ = oracle.attention_bwd_rows(qb, kb, vb, dob, dtype, scale, causal, np.zeros(rows.size, np.int64),
                                              rows)
        dk_ref, dv_ref = oracle.attention_bwd_keys(qb, kb, vb, dob, dtype, scale, causal, 0, keys)
        ir, ik = torch.from_numpy(rows).cuda(), torch.from_numpy(keys).cuda()
        got = [dq[b, h, ir], dk[b, h, ik], dv[b, h, ik]]
        got = [g.double().cpu().numpy() for g in got]
        common = max(float(np.abs(r).max()) for r in (dq_ref, dk_ref, dv_ref))
        label = "B%d H%d N%d d%d head (%d, %d)" % (B, H, N, d, b, h)
        for name, g, r in zip(("dQ rows", "dK last keys", "dV last keys"), got, (dq_ref, dk_ref, dv_ref)):
            grad_check(g, r, dtype, label + " " + name, common)
    del q, k, v, dout, dq, dk, dv
    torch.cuda.empty_cache()
