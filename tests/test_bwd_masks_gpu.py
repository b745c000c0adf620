"""Parity of the general backward pass (fa2_bwd_ex: band and prefix masks,
N_q != N_k, strided layouts, packed batches) with the oracle's masked
backward, through the C ABI.

Each gradient is compared against its own scale, as for the square backward:
max|g - g_oracle| <= TOL * max|g_oracle| (floored at 1e-3 of the largest
gradient's scale), TOL 3e-3 (fp16) / 1.5e-2 (bf16).  Keys no query row sees
must get dK = dV = 0 exactly, query rows that see no key dQ = 0 exactly.
Layout changes only change addressing; dK and dV (each written once) are
then bit-identical to the contiguous call, dQ (fp32 reduce-adds in L2) within
a few units of its last place.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
import oracle
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu

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


def status_ok():
    torch.cuda.synchronize()
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_OK, "device status 0x%x" % detail


def inputs(B, H, Nq, Nk, d, dtype, seed):
    q = sy.make_qkv(B, H, Nq, d, dtype, seed)[0]
    _, k, v = sy.make_qkv(B, H, Nk, d, dtype, seed + 1)
    do = sy.make_qkv(B, H, Nq, d, dtype, seed + 2)[0]
    return q, k, v, do


def visible(Nq, Nk, wl, wr, pre):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    off = Nk - Nq
    band = np.ones((Nq, Nk), dtype=bool)
    if wl >= 0:
        band &= j >= i + off - wl
    if wr >= 0:
        band &= j <= i + off + wr
    return band | (j < pre)


def check(got, ref, dtype, label, vis=None):
    common = max(float(np.abs(r).max()) for r in ref[:3])
    if vis is not None:   # gradients of rows / keys no visible pair touches are exactly 0
        assert np.all(got[0][..., ~vis.any(axis=1), :] == 0), label + ": dQ of a row without keys"
        assert np.all(got[1][..., ~vis.any(axis=0), :] == 0), label + ": dK of a key nobody sees"
        assert np.all(got[2][..., ~vis.any(axis=0), :] == 0), label + ": dV of a key nobody sees"
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref[:3]):
        assert np.isfinite(g).all(), "%s %s: non-finite" % (label, name)
        den = max(float(np.abs(r).max()), 1e-3 * common, 1e-30)
        rel = float(np.abs(g - r).max() / den)
        print("%s %s: max|err|/max|ref| = %.3e" % (label, name, rel))
        assert rel <= TOL[dtype], "%s %s: %.3e > %.0e" % (label, name, rel, TOL[dtype])


def run(q, k, v, do, dtype, scale, **mask):
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = fa2.fa2_fwd_ex(tq, tk, tv, scale=scale, **mask)
    dq, dk, dv = fa2.fa2_bwd_ex(tq, tk, tv, o, lse, tdo, scale=scale, **mask)
    status_ok()
    return [g.double().cpu().numpy() for g in (dq, dk, dv)]


SHAPES = [(1, 1), (64, 200), (200, 64), (129, 129), (300, 700), (700, 300)]
MASKS = [(-1, -1, 0), (-1, 0, 0), (0, 0, 0), (40, 0, 0), (100, 30, 0), (200, -1, 0), (-1, 0, 70), (5, 0, 150)]


@pytest.mark.parametrize("d,dtype", [(64, sy.FP16), (128, sy.BF16), (128, sy.FP16), (256, sy.FP16), (256, sy.BF16)])
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", SHAPES)
def test_bwd_masks(Nq, Nk, mask, d, dtype):
    wl, wr, pre = mask
    q, k, v, do = inputs(1, 2, Nq, Nk, d, dtype, seed=15000 + Nq + 3 * Nk + d)
    scale = 1.0 / np.sqrt(d)
    got = run(q, k, v, do, dtype, scale, window_left=wl, window_right=wr, prefix_len=pre)
    ref = oracle.attention_bwd_masked(q, k, v, do, dtype, scale, wl, wr, pre)
    check(got, ref, dtype, "Nq=%d Nk=%d mask=%s d=%d" % (Nq, Nk, mask, d), visible(Nq, Nk, wl, wr, pre))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bwd_bnhd_views(d):
    """q, k, v, o, dout and the gradients as [B, N, H, d] views: dK and dV
    bit-identical to the contiguous call, dQ within fp32 reduce-add rounding."""
    B, H, Nq, Nk, dtype = 2, 3, 300, 500, sy.BF16
    q, k, v, do = inputs(B, H, Nq, Nk, d, dtype, seed=15500 + d)
    mask = dict(window_left=64, window_right=0)
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = fa2.fa2_fwd_ex(tq, tk, tv, **mask)
    g1 = fa2.fa2_bwd_ex(tq, tk, tv, o, lse, tdo, **mask)
    view = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)
    bq, bk, bv, bo, bdo = (view(t) for t in (tq, tk, tv, o, tdo))
    g2 = fa2.fa2_bwd_ex(bq, bk, bv, bo, lse, bdo, **mask)
    status_ok()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert torch.allclose(g1[0].float(), g2[0].float(), rtol=2 ** -7, atol=1e-3)
    ref = oracle.attention_bwd_masked(q, k, v, do, dtype, 1.0 / np.sqrt(d), 64, 0, 0)
    check([g.double().cpu().numpy() for g in g2], ref, dtype, "bnhd d=%d" % d)


@pytest.mark.parametrize("d", [128, 256])
def test_bwd_packed_sequences(d):
    """Packed sequences of mixed lengths (one without keys, one without
    queries): each sequence's gradients match the oracle on its slice; dq rows
    outside every sequence are zero."""
    H, dtype = 2, sy.BF16
    lens_q = [1, 129, 0, 300, 64, 200]
    lens_k = [1, 200, 5, 300, 0, 513]
    mask = dict(window_left=-1, window_right=0)
    seqs = [inputs(1, H, max(nq, 1), max(nk, 1), d, dtype, seed=15700 + 9 * i)
            for i, (nq, nk) in enumerate(zip(lens_q, lens_k))]
    tail = 7
    pack = lambda xs: np.ascontiguousarray(np.concatenate(xs, axis=0))
    qp = pack([s[0][0].transpose(1, 0, 2)[:nq] for s, nq in zip(seqs, lens_q)] + [np.zeros((tail, H, d), np.uint16)])
    dop = pack([s[3][0].transpose(1, 0, 2)[:nq] for s, nq in zip(seqs, lens_q)] + [np.zeros((tail, H, d), np.uint16)])
    kp = pack([s[1][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, lens_k)])
    vp = pack([s[2][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, lens_k)])
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32, device="cuda")
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (qp, kp, vp, dop))
    pk = dict(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=max(lens_q))
    o, lse = fa2.fa2_fwd_ex(tq, tk, tv, **mask, **pk)
    dq, dk, dv = fa2.fa2_bwd_ex(tq, tk, tv, o, lse, tdo, **mask, **pk, max_seqlen_k=max(lens_k))
    status_ok()
    assert torch.all(dq[sum(lens_q):] == 0)
    rq = rk = 0
    for i, (nq, nk) in enumerate(zip(lens_q, lens_k)):
        if nq and nk:
            q, k, v, do = (np.ascontiguousarray(x) for x in seqs[i])
            k, v = np.ascontiguousarray(k[:, :, :nk]), np.ascontiguousarray(v[:, :, :nk])
            ref = oracle.attention_bwd_masked(q[:, :, :nq].copy(), k, v, do[:, :, :nq].copy(), dtype,
                                              1.0 / np.sqrt(d), -1, 0, 0)
            got = [dq[rq:rq + nq].permute(1, 0, 2).unsqueeze(0), dk[rk:rk + nk].permute(1, 0, 2).unsqueeze(0),
                   dv[rk:rk + nk].permute(1, 0, 2).unsqueeze(0)]
            check([g.double().cpu().numpy() for g in got], ref, dtype, "seq %d" % i)
        elif nk:   # keys no query sees
            assert torch.all(dk[rk:rk + nk] == 0) and torch.all(dv[rk:rk + nk] == 0)
        elif nq:   # queries without keys
            assert torch.all(dq[rq:rq + nq] == 0)
        rq += nq
        rk += nk


@pytest.mark.parametrize("d,dtype,nseq", [(64, sy.FP16, 192), (128, sy.BF16, 192), (128, sy.BF16, 193),
                                          (256, sy.FP16, 192), (256, sy.BF16, 193)])
def test_bwd_packed_many_sequences(d, dtype, nseq):
    """192 packed sequences (the grid holds one CTA per real key tile, each
    finding its sequence from the offsets) and 193 (one CTA per sequence,
    head and key tile of the longest), some empty: each sequence's gradients
    match the oracle on its slice."""
    H, wl, wr = 2, -1, 0
    rng = np.random.default_rng(15800 + nseq + d)
    lens = rng.integers(1, 300, nseq)
    lens[::17] = 0
    lens[7] = 300
    total = int(lens.sum())
    q, k, v, do = inputs(1, H, total, total, d, dtype, seed=15810 + nseq + d)
    packed = [to_dev(np.ascontiguousarray(x[0].transpose(1, 0, 2)), dtype) for x in (q, k, v, do)]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    pk = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=int(lens.max()), window_left=wl, window_right=wr)
    o, lse = fa2.fa2_fwd_ex(packed[0], packed[1], packed[2], **pk)
    grads = fa2.fa2_bwd_ex(packed[0], packed[1], packed[2], o, lse, packed[3], **pk, max_seqlen_k=int(lens.max()))
    status_ok()
    grads = [g.double().cpu().numpy() for g in grads]
    row = 0
    for i, n in enumerate(lens.tolist()):
        if n:
            sl = lambda x: np.ascontiguousarray(x[:, :, row:row + n])
            ref = oracle.attention_bwd_masked(sl(q), sl(k), sl(v), sl(do), dtype, 1.0 / np.sqrt(d), wl, wr, 0)
            got = [g[row:row + n].transpose(1, 0, 2)[None] for g in grads]
            check(got, ref, dtype, "seq %d of %d (n=%d)" % (i, nseq, n))
        row += n


@pytest.mark.parametrize("trial", range(4))
def test_bwd_packed_random_mixes_match_unpacked(trial):
    """Random packed batches (up to 200 sequences, skewed lengths, empty ones,
    N_q != N_k): each sequence's dK and dV bit-equal the unpacked call on that
    sequence alone (summed inside one CTA in a fixed order), dQ equals it to
    rounding (fp32 reduce-adds land in run-dependent order), and dq rows
    outside every sequence are zero."""
    rng = np.random.default_rng(15900 + trial)
    nseq = int(rng.choice([3, 40, 192, 200]))
    d, dtype = [(64, sy.FP16), (128, sy.BF16)][trial % 2]
    H = int(rng.integers(1, 3))
    wl, wr = [(-1, 0), (-1, -1), (int(rng.integers(0, 300)), 0), (-1, 0)][trial]
    top = 1500 if nseq <= 40 else 300
    lq = np.minimum(rng.exponential(top / 4, nseq).astype(np.int64), top)
    lk = np.where(rng.random(nseq) < 0.5, lq, np.minimum(rng.exponential(top / 4, nseq).astype(np.int64), top))
    lq[rng.random(nseq) < 0.1] = 0
    lq[0], lk[0] = max(int(lq[0]), 1), max(int(lk[0]), 1)
    tq, tk, tail = int(lq.sum()), int(lk.sum()), 3
    q, k, v, do = inputs(1, H, tq + tail, tk, d, dtype, seed=15910 + trial)
    tq_, tk_, tv_, tdo_ = (to_dev(np.ascontiguousarray(x[0].transpose(1, 0, 2)), dtype) for x in (q, k, v, do))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32, device="cuda")
    mask = dict(window_left=wl, window_right=wr)
    pk = dict(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=int(lq.max()))
    o, lse = fa2.fa2_fwd_ex(tq_, tk_, tv_, **mask, **pk)
    dq, dk, dv = fa2.fa2_bwd_ex(tq_, tk_, tv_, o, lse, tdo_, **mask, **pk, max_seqlen_k=int(lk.max()))
    status_ok()
    assert torch.all(dq[tq:] == 0)
    view = lambda x, a, n: x[a:a + n].permute(1, 0, 2).unsqueeze(0)
    rq = rk = 0
    for i, (nq, nk) in enumerate(zip(lq.tolist(), lk.tolist())):
        label = "trial %d seq %d of %d (nq=%d nk=%d) d=%d" % (trial, i, nseq, nq, nk, d)
        if nq and nk:
            sq, sk, sv, sdo = view(tq_, rq, nq), view(tk_, rk, nk), view(tv_, rk, nk), view(tdo_, rq, nq)
            ou, lu = fa2.fa2_fwd_ex(sq, sk, sv, **mask)
            gu = fa2.fa2_bwd_ex(sq, sk, sv, ou, lu, torch.empty_like(ou).copy_(sdo), **mask)   # dout in o's layout
            status_ok()
            assert torch.equal(view(dk, rk, nk), gu[1]) and torch.equal(view(dv, rk, nk), gu[2]), label + ": dK / dV"
            ref = gu[0].float()
            err = float((view(dq, rq, nq).float() - ref).abs().max())
            assert err <= 1e-2 * max(float(ref.abs().max()), 1e-6), label + ": dQ %.3e" % err
        elif nk:
            assert torch.all(dk[rk:rk + nk] == 0) and torch.all(dv[rk:rk + nk] == 0), label
        elif nq:
            assert torch.all(dq[rq:rq + nq] == 0), label
        rq += nq
        rk += nk


@pytest.mark.parametrize("Nq,Nk,mask,d,dtype", [
    (2048, 8192, (-1, 0, 0), 128, sy.BF16),     # a query chunk at the end of a long key sequence
    (4096, 4096, (511, 0, 0), 64, sy.FP16),     # sliding window of 512 keys
    (3000, 3000, (-1, 0, 1000), 128, sy.BF16),  # prefix-LM
    (1500, 3000, (-1, 0, 0), 256, sy.FP16),     # d = 256: a query chunk after a key prefix
])
def test_bwd_masks_larger(Nq, Nk, mask, d, dtype):
    wl, wr, pre = mask
    q, k, v, do = inputs(1, 2, Nq, Nk, d, dtype, seed=15900 + Nq)
    scale = 1.0 / np.sqrt(d)
    got = run(q, k, v, do, dtype, scale, window_left=wl, window_right=wr, prefix_len=pre)
    ref = oracle.attention_bwd_masked(q, k, v, do, dtype, scale, wl, wr, pre)
    check(got, ref, dtype, "Nq=%d Nk=%d mask=%s" % (Nq, Nk, mask), visible(Nq, Nk, wl, wr, pre))
