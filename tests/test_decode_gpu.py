"""Parity of the decoding-regime kernel (fa2_decode: at most 8 query rows
per sequence, keys split across CTAs and merged) with the CPU oracle, through
the C ABI.

Tolerances as for the forward pass: max |O_gpu - O_oracle| <= 2e-3 (fp16) or
1e-2 (bf16) and max |LSE_gpu - LSE_oracle| <= 1e-3 on rows that see a key;
rows that see none must be exactly O = 0 and LSE = -inf.
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


def qkv(B, H, Nq, Nk, d, dtype, seed):
    q = sy.make_qkv(B, H, Nq, d, dtype, seed)[0]
    _, k, v = sy.make_qkv(B, H, Nk, d, dtype, seed + 1)
    return q, k, v


def status_ok():
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "device status 0x%x" % detail


def check(o, lse, o_ref, lse_ref, dtype, label):
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), label + ": rows without keys differ"
    assert np.all(o[empty] == 0), label + ": a row without keys is not zero"
    full = ~empty
    if not full.any():
        return
    og, orf, lg, lrf = o[full], o_ref[full], lse[full], lse_ref[full]
    assert np.isfinite(og).all() and np.isfinite(lg).all(), label + ": non-finite output"
    eo = float(np.abs(og - orf).max())
    el = float(np.abs(lg - lrf).max())
    print("%s: max|dO| %.3e (tol %.0e)  max|dLSE| %.3e" % (label, eo, TOL_O[dtype], el))
    assert eo <= TOL_O[dtype], "%s: O error %.3e" % (label, eo)
    assert el <= TOL_LSE, "%s: LSE error %.3e" % (label, el)


def run_decode(q, k, v, dtype, scale, **kw):
    o, lse = fa2.fa2_decode(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, **kw)
    status_ok()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


MASKS = [(-1, -1, 0), (-1, 0, 0), (100, 0, 0), (0, 0, 0), (64, 0, 5), (2, 3, 0)]


@pytest.mark.parametrize("d,dtype", [(64, sy.FP16), (128, sy.BF16), (256, sy.BF16), (128, sy.FP16)])
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("nq,nk", [(1, 1), (1, 63), (1, 65), (2, 300), (3, 4097), (5, 1000), (8, 2500), (8, 3)])
def test_decode_all_outputs(nq, nk, mask, d, dtype):
    wl, wr, pre = mask
    q, k, v = qkv(2, 3, nq, nk, d, dtype, seed=12000 + 7 * nq + nk + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_decode(q, k, v, dtype, scale, window_left=wl, window_right=wr, prefix_len=pre)
    o_ref, lse_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_left=wl, window_right=wr,
                                                 prefix_len=pre)
    check(o, lse, o_ref, lse_ref, dtype, "nq=%d nk=%d mask=%s d=%d" % (nq, nk, mask, d))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_bnhd_cache_equals_contiguous(d):
    """K/V as [B, N, H, d] caches (strided views): bit-identical to the contiguous call."""
    B, H, nq, nk, dtype = 2, 4, 2, 3000, sy.BF16
    q, k, v = qkv(B, H, nq, nk, d, dtype, seed=12500 + d)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o1, l1 = fa2.fa2_decode(qd, kd, vd, window_left=-1, window_right=0)
    kb, vb = (x.transpose(1, 2).contiguous().transpose(1, 2) for x in (kd, vd))
    o2, l2 = fa2.fa2_decode(qd, kb, vb, window_left=-1, window_right=0)
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_packed_caches():
    """One new token per sequence against caches of mixed lengths (one empty,
    one with two query rows), packed: each equals the oracle on its slice."""
    H, d, dtype = 4, 128, sy.BF16
    lens_k = [1, 700, 0, 5000, 129, 64, 2049]
    lens_q = [1, 1, 1, 2, 1, 1, 1]
    seqs = [qkv(1, H, nq, max(nk, 1), d, dtype, seed=12600 + 5 * i) for i, (nq, nk) in enumerate(zip(lens_q, lens_k))]
    qp = np.concatenate([s[0][0].transpose(1, 0, 2) for s in seqs], axis=0)
    kp = np.concatenate([s[1][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, lens_k)], axis=0)
    vp = np.concatenate([s[2][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, lens_k)], axis=0)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    o, lse = fa2.fa2_decode(to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype), window_left=-1,
                            window_right=0, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=2,
                            max_seqlen_k=max(lens_k))
    status_ok()
    row = 0
    for i, (nq, nk) in enumerate(zip(lens_q, lens_k)):
        og = o[row:row + nq].permute(1, 0, 2).unsqueeze(0).double().cpu().numpy()
        lg = lse[:, row:row + nq].unsqueeze(0).double().cpu().numpy()
        if nk == 0:
            assert np.all(og == 0) and np.all(np.isneginf(lg))
        else:
            qs = np.ascontiguousarray(seqs[i][0])
            ks, vs = (np.ascontiguousarray(x[:, :, :nk]) for x in seqs[i][1:])
            o_ref, l_ref = oracle.attention_fwd_masked(qs, ks, vs, dtype, 1.0 / np.sqrt(d), window_left=-1,
                                                       window_right=0)
            check(og, lg, o_ref, l_ref, dtype, "seq %d nk=%d" % (i, nk))
        row += nq


@pytest.mark.parametrize("rows", [1, 2])
def test_decode_sequence_longer_than_plan_is_reported(rows):
    """A packed sequence with more keys than max_seqlen_k lets the split plan
    cover is reported and left unwritten, on both paths (one row: CUDA-core
    kernel; two rows: tensor-core kernel)."""
    H, d, dtype = 2, 64, sy.FP16
    q, k, v = qkv(1, H, 2 * rows, 900, d, dtype, seed=12700 + rows)
    qp, kp, vp = (np.ascontiguousarray(x[0].transpose(1, 0, 2)) for x in (q, k, v))
    cu_q = torch.tensor([0, rows, 2 * rows], dtype=torch.int32, device="cuda")
    cu_k = torch.tensor([0, 300, 900], dtype=torch.int32, device="cuda")   # second sequence: 600 keys
    o = torch.full((2 * rows, H, d), 3.0, dtype=torch.float16, device="cuda")
    lse = torch.full((H, 2 * rows), 4.0, dtype=torch.float32, device="cuda")
    fa2.fa2_decode(to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype), o=o, lse=lse, cu_seqlens_q=cu_q,
                   cu_seqlens_k=cu_k, max_seqlen_q=rows, max_seqlen_k=300)
    torch.cuda.synchronize()
    code, _ = fa2.fa2_get_device_status()
    assert code == fa2.FA2_ERR_DEVICE_SEQLENS
    assert torch.all(o[rows:] == 3.0) and torch.all(lse[:, rows:] == 4.0)    # the long one is left as it was
    assert not torch.any(o[:rows] == 3.0)


@pytest.mark.parametrize("nk,d,dtype", [(131072, 128, sy.BF16), (65536, 64, sy.FP16), (32768, 256, sy.BF16)])
def test_decode_long_caches(nk, d, dtype):
    B, H = 1, 8
    q, k, v = qkv(B, H, 1, nk, d, dtype, seed=12800 + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_decode(q, k, v, dtype, scale, window_left=-1, window_right=0)
    o_ref, l_ref = oracle.attention_rows_masked(q, k, v, dtype, scale, np.arange(B * H), np.zeros(B * H, np.int64),
                                                window_left=-1, window_right=0)
    check(o.reshape(B * H, d), lse.reshape(B * H), o_ref, l_ref, dtype, "nk=%d d=%d" % (nk, d))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_tensor_core_path_bnhd_equals_contiguous(d):
    """Six rows (the tensor-core split path): K/V as [B, N, H, d] views give
    bit-identical results to contiguous caches, and both equal the oracle."""
    B, H, nq, nk, dtype = 2, 3, 6, 5000, sy.BF16
    q, k, v = qkv(B, H, nq, nk, d, dtype, seed=13000 + d)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o1, l1 = fa2.fa2_decode(qd, kd, vd, window_left=-1, window_right=0)
    kb, vb = (x.transpose(1, 2).contiguous().transpose(1, 2) for x in (kd, vd))
    o2, l2 = fa2.fa2_decode(qd, kb, vb, window_left=-1, window_right=0)
    status_ok()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    scale = 1.0 / np.sqrt(d)
    o_ref, lse_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_left=-1, window_right=0)
    check(o1.double().cpu().numpy(), l1.double().cpu().numpy(), o_ref, lse_ref, dtype, "tensor-core path d=%d" % d)


@pytest.mark.parametrize("nq", [3, 8])
def test_decode_tensor_core_path_long_cache(nq):
    """Several rows against a 65536-key cache: dozens of key chunks per
    (b, h) on the tensor-core path, every row checked against the oracle."""
    B, H, nk, d, dtype = 1, 8, 65536, 128, sy.BF16
    q, k, v = qkv(B, H, nq, nk, d, dtype, seed=13100 + nq)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_decode(q, k, v, dtype, scale, window_left=-1, window_right=0)
    bh = np.repeat(np.arange(B * H), nq)
    rows = np.tile(np.arange(nq), B * H)
    o_ref, l_ref = oracle.attention_rows_masked(q, k, v, dtype, scale, bh, rows, window_left=-1, window_right=0)
    check(o.reshape(B * H * nq, d), lse.reshape(B * H * nq), o_ref, l_ref, dtype, "nq=%d nk=%d" % (nq, nk))


@pytest.mark.parametrize("nq", [1, 4])
def test_decode_window_chunks_start_at_the_band(nq):
    """A bounded window against a long cache: the key chunks cover only the
    band the rows see (both the CUDA-core and the tensor-core path)."""
    B, H, nk, d, dtype = 1, 4, 20000, 128, sy.BF16
    q, k, v = qkv(B, H, nq, nk, d, dtype, seed=13200 + nq)
    scale = 1.0 / np.sqrt(d)
    for wl in (1000, 4095):
        o, lse = run_decode(q, k, v, dtype, scale, window_left=wl, window_right=0)
        o_ref, l_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_left=wl, window_right=0)
        check(o, lse, o_ref, l_ref, dtype, "nq=%d window %d" % (nq, wl))


def test_decode_repeated_calls_bit_identical():
    q, k, v = qkv(4, 8, 4, 20000, 128, sy.BF16, seed=12900)
    qd, kd, vd = (to_dev(x, sy.BF16) for x in (q, k, v))
    ws = torch.empty(fa2.fa2_decode_workspace_bytes(qd, kd, vd), dtype=torch.uint8, device="cuda")
    first = fa2.fa2_decode(qd, kd, vd, workspace=ws, window_left=4096, window_right=0)
    for _ in range(3):
        again = fa2.fa2_decode(qd, kd, vd, workspace=ws, window_left=4096, window_right=0)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    status_ok()
