"""The forward pass on tensors past 2^31 elements (4 GiB each), against the oracle.

Element offsets of the last heads' rows exceed 32 bits there, and the row
coordinates reach 262143, so any 32-bit product in the index arithmetic of the
kernels or the host (tensor maps, the LSE and O row offsets, the grid) shows
up as a wrong or missing row.  The inputs are drawn on the device from a seeded
generator (N(0, 1) in fp32, rounded once to the 16-bit type), one head at a
time; the oracle recomputes sampled rows of the first and the last heads from
those heads' own inputs copied back to the host.

Tolerances as in test_parity_gpu: max |O - O_oracle| <= 2e-3 (fp16) or 1e-2
(bf16) and max |LSE - LSE_oracle| <= 1e-3.
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
