"""Kernels launched concurrently on separate streams share SMs: the forward
kernel runs two CTAs per SM with 256 TMEM columns each, the backward kernel
takes all 512 columns of an SM, the decode path 256.  A CTA whose TMEM
allocation finds the columns taken waits until their holder exits, and no
holder waits on anything outside its own CTA.  These tests overlap the three
paths on three streams many times and require each result to equal the same
call run alone: bit for bit, except the backward's dQ, whose fp32 sums over
key tiles land in run-dependent order (within rounding)."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa2_build.build()
    fa2.load_library()


def to_dev(bits, dtype):
    tdt = torch.bfloat16 if dtype == sy.BF16 else torch.float16
    return torch.from_numpy(bits.view(np.int16)).view(tdt).cuda()


def test_forward_backward_decode_overlapped_on_three_streams():
    dt = sy.BF16
    # forward + backward problem (d = 128, causal) and a decode problem (4 rows)
    q, k, v = (to_dev(x, dt) for x in sy.make_qkv(2, 8, 2048, 128, dt, seed=14000))
    dout = to_dev(sy.make_qkv(2, 8, 2048, 128, dt, seed=14001)[0], dt)
    qd = to_dev(sy.make_qkv(2, 8, 4, 128, dt, seed=14002)[0], dt)
    kc, vc = (to_dev(x, dt) for x in sy.make_qkv(2, 8, 8192, 128, dt, seed=14003)[1:])
    ws_b = torch.empty(fa2.fa2_bwd_workspace_bytes(2, 8, 2048, 128), dtype=torch.uint8, device="cuda")
    ws_d = torch.empty(fa2.fa2_decode_workspace_bytes(qd, kc, vc), dtype=torch.uint8, device="cuda")

    # each call alone
    o_ref, l_ref = fa2.fa2_fwd(q, k, v, causal=True)
    g_ref = fa2.fa2_bwd(q, k, v, o_ref, l_ref, dout, workspace=ws_b, causal=True)
    d_ref = fa2.fa2_decode(qd, kc, vc, workspace=ws_d, window_left=-1, window_right=0)
    torch.cuda.synchronize()

    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    o, lse = torch.empty_like(o_ref), torch.empty_like(l_ref)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    od, ld = torch.empty_like(d_ref[0]), torch.empty_like(d_ref[1])
    for _ in range(20):
        fa2.fa2_fwd(q, k, v, o, lse, causal=True, stream=s1)
        fa2.fa2_bwd(q, k, v, o_ref, l_ref, dout, dq, dk, dv, ws_b, causal=True, stream=s2)
        fa2.fa2_decode(qd, kc, vc, od, ld, ws_d, window_left=-1, window_right=0, stream=s3)
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "device status 0x%x" % detail
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), "forward differs"
    assert torch.equal(od, d_ref[0]) and torch.equal(ld, d_ref[1]), "decode differs"
    # dK and dV are summed inside one CTA in a fixed order; dQ by fp32 reduce-adds
    # from many CTAs in the order they land, so only to rounding
    assert torch.equal(dk, g_ref[1]) and torch.equal(dv, g_ref[2]), "dK / dV differ"
    scale = g_ref[0].float().abs().max().item()
    err = (dq.float() - g_ref[0].float()).abs().max().item()
    assert err <= 1e-2 * scale, "dQ differs beyond rounding: %.3e of %.3e" % (err, scale)
