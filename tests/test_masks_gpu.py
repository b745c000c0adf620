"""Parity of the general forward pass (fa2_fwd_ex: band and prefix masks,
N_q != N_k, strided layouts, packed variable-length batches) with the CPU
oracle, through the C ABI.

Tolerances as for the square forward pass: max |O_gpu - O_oracle| <= 2e-3
(fp16) or 1e-2 (bf16) and max |LSE_gpu - LSE_oracle| <= 1e-3 on rows that
see at least one key; rows that see none must be exactly O = 0 and
LSE = -inf.  Layout changes (strides, packing) only change addressing, so
those results must also be bit-identical to the contiguous call.
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
    print("%s: max|dO| %.3e (tol %.0e)  max|dLSE| %.3e  empty rows %d" % (label, eo, TOL_O[dtype], el, empty.sum()))
    assert eo <= TOL_O[dtype], "%s: O error %.3e" % (label, eo)
    assert el <= TOL_LSE, "%s: LSE error %.3e" % (label, el)


def run_ex(q, k, v, dtype, scale, **mask):
    o, lse = fa2.fa2_fwd_ex(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, **mask)
    status_ok()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


# ------------------------------------------------------------------ masks x lengths, every output

SHAPES = [(1, 1), (64, 200), (200, 64), (129, 129), (300, 1000), (1000, 300), (384, 384)]
MASKS = [  # (window_left, window_right, prefix_len)
    (-1, -1, 0), (-1, 0, 0), (0, 0, 0), (16, 0, 0), (100, 50, 0), (0, -1, 0), (200, -1, 0), (-1, 0, 40),
    (5, 0, 130), (-1, 7, 0), (2 ** 31 - 1, 0, 0),
]
KINDS = [(64, sy.BF16), (128, sy.FP16), (128, sy.BF16), (256, sy.BF16)]


@pytest.mark.parametrize("d,dtype", KINDS)
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Nq,Nk", SHAPES)
def test_masks_all_outputs(Nq, Nk, mask, d, dtype):
    wl, wr, pre = mask
    q, k, v = qkv(1, 2, Nq, Nk, d, dtype, seed=9000 + Nq + 7 * Nk + d)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_ex(q, k, v, dtype, scale, window_left=wl, window_right=wr, prefix_len=pre)
    o_ref, lse_ref = oracle.attention_fwd_masked(q, k, v, dtype, scale, window_left=wl, window_right=wr,
                                                 prefix_len=pre)
    check(o, lse, o_ref, lse_ref, dtype, "Nq=%d Nk=%d mask=%s d=%d" % (Nq, Nk, mask, d))


def test_causal_window_equals_fa2_fwd_causal():
    q, k, v = qkv(2, 3, 700, 700, 128, sy.BF16, seed=9100)
    qd, kd, vd = (to_dev(x, sy.BF16) for x in (q, k, v))
    a = fa2.fa2_fwd(qd, kd, vd, causal=True)
    b = fa2.fa2_fwd_ex(qd, kd, vd, window_left=-1, window_right=0)
    status_ok()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# ------------------------------------------------------------------ strided layouts

@pytest.mark.parametrize("d,dtype", [(64, sy.FP16), (128, sy.BF16), (256, sy.FP16)])
@pytest.mark.parametrize("mask", [(-1, 0, 0), (48, 0, 0), (-1, -1, 0)])
def test_bnhd_views_and_packed_qkv_bit_identical(d, dtype, mask):
    """q, k, v as [B,N,H,d] tensors (transposed views), as slices of one packed
    [B,N,3,H,d] QKV tensor, o written into a [B,N,H,d] view and lse into a
    [H,B,N] tensor: bit-identical to the contiguous call, and nothing outside
    the output views is touched."""
    B, H, Nq, Nk = 2, 3, 333, 333
    wl, wr, pre = mask
    q, k, v = qkv(B, H, Nq, Nk, d, dtype, seed=9200 + d)
    qd, kd, vd = (to_dev(x, dtype) for x in (q, k, v))
    o_ref, l_ref = fa2.fa2_fwd_ex(qd, kd, vd, window_left=wl, window_right=wr, prefix_len=pre)
    # [B, N, H, d] storage, passed as [B, H, N, d] views
    qb, kb, vb = (x.transpose(1, 2).contiguous().transpose(1, 2) for x in (qd, kd, vd))
    assert qb.stride() == (Nq * H * d, d, H * d, 1)
    ob = torch.full((B, Nq, H, d), 7.0, dtype=qd.dtype, device="cuda").transpose(1, 2)
    lb = torch.full((H, B, Nq), 9.0, dtype=torch.float32, device="cuda").transpose(0, 1)
    fa2.fa2_fwd_ex(qb, kb, vb, o=ob, lse=lb, window_left=wl, window_right=wr, prefix_len=pre)
    status_ok()
    assert torch.equal(ob, o_ref) and torch.equal(lb, l_ref)
    # one packed [B, N, 3, H, d] tensor, output into a padded buffer
    qkv_packed = torch.stack([qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2)], dim=2).contiguous()
    qp, kp, vp = (qkv_packed[:, :, i].transpose(1, 2) for i in range(3))
    pad = torch.full((B, H, Nq, d + 64), 5.0, dtype=qd.dtype, device="cuda")
    op = pad[..., :d]
    fa2.fa2_fwd_ex(qp, kp, vp, o=op, window_left=wl, window_right=wr, prefix_len=pre)
    status_ok()
    assert torch.equal(op, o_ref)
    assert torch.all(pad[..., d:] == 5.0)
    # and against the oracle
    o_orc, l_orc = oracle.attention_fwd_masked(q, k, v, dtype, 1.0 / np.sqrt(d), window_left=wl, window_right=wr,
                                               prefix_len=pre)
    check(o_ref.double().cpu().numpy(), l_ref.double().cpu().numpy(), o_orc, l_orc, dtype, "bnhd d=%d" % d)


# ------------------------------------------------------------------ packed variable-length batches

LENS_Q = [1, 127, 128, 129, 300, 0, 57, 513]
LENS_K = [1, 200, 128, 64, 300, 5, 0, 513]


def _pack(seqs):
    return np.ascontiguousarray(np.concatenate(seqs, axis=0)) if seqs else None


@pytest.mark.parametrize("d,dtype", [(64, sy.BF16), (128, sy.FP16), (256, sy.BF16)])
@pytest.mark.parametrize("mask", [(-1, 0, 0), (32, 0, 0), (-1, -1, 0), (-1, 0, 20)])
def test_packed_sequences(d, dtype, mask):
    """Sequences of mixed lengths (including an empty one and one without
    keys) packed as [total, H, d]: each equals the oracle on its own slice,
    and bit-equals the unpacked call on that sequence alone; padding rows
    after the last sequence stay untouched."""
    wl, wr, pre = mask
    H = 2
    scale = 1.0 / np.sqrt(d)
    seqs = [qkv(1, H, max(nq, 1), max(nk, 1), d, dtype, seed=9300 + 11 * i + d)
            for i, (nq, nk) in enumerate(zip(LENS_Q, LENS_K))]
    # [1, H, n, d] -> [n, H, d]
    q_rows = [s[0][0].transpose(1, 0, 2)[:nq] for s, nq in zip(seqs, LENS_Q)]
    k_rows = [s[1][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, LENS_K)]
    v_rows = [s[2][0].transpose(1, 0, 2)[:nk] for s, nk in zip(seqs, LENS_K)]
    tail = 9  # padding rows after the last sequence
    qp = _pack(q_rows + [np.zeros((tail, H, d), np.uint16)])
    kp, vp = _pack(k_rows), _pack(v_rows)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(LENS_Q)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(LENS_K)]), dtype=torch.int32, device="cuda")
    qd, kd, vd = to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype)
    o = torch.full(qd.shape, 3.0, dtype=qd.dtype, device="cuda")
    lse = torch.full((H, qd.shape[0]), 4.0, dtype=torch.float32, device="cuda")
    fa2.fa2_fwd_ex(qd, kd, vd, o=o, lse=lse, window_left=wl, window_right=wr, prefix_len=pre, cu_seqlens_q=cu_q,
                   cu_seqlens_k=cu_k, max_seqlen_q=max(LENS_Q))
    status_ok()
    total = int(sum(LENS_Q))
    assert torch.all(o[total:] == 3.0) and torch.all(lse[:, total:] == 4.0)
    row = 0
    for i, (nq, nk) in enumerate(zip(LENS_Q, LENS_K)):
        if nq == 0:
            continue
        og = o[row:row + nq].permute(1, 0, 2).unsqueeze(0)        # [1, H, nq, d]
        lg = lse[:, row:row + nq].unsqueeze(0)                     # [1, H, nq]
        label = "seq %d (nq=%d nk=%d) mask=%s d=%d" % (i, nq, nk, mask, d)
        if nk == 0:
            assert torch.all(og == 0) and torch.all(torch.isneginf(lg)), label
        else:
            qs = np.ascontiguousarray(seqs[i][0][:, :, :nq])
            ks, vs = (np.ascontiguousarray(x[:, :, :nk]) for x in seqs[i][1:])
            ou, lu = fa2.fa2_fwd_ex(to_dev(qs, dtype), to_dev(ks, dtype), to_dev(vs, dtype), window_left=wl,
                                    window_right=wr, prefix_len=pre)
            status_ok()
            assert torch.equal(og, ou) and torch.equal(lg, lu), label + ": packed != unpacked"
            o_orc, l_orc = oracle.attention_fwd_masked(qs, ks, vs, dtype, scale, window_left=wl, window_right=wr,
                                                       prefix_len=pre)
            check(og.double().cpu().numpy(), lg.double().cpu().numpy(), o_orc, l_orc, dtype, label)
        row += nq


def _tile_search_grid(lens, rows=128):
    """Whether the host sizes a packed batch's grid to its real tiles (each
    CTA then finds its sequence and tile from the offsets): at most 192
    sequences, and fewer tiles than one per sequence, head and tile of the
    longest sequence."""
    B, total = len(lens), int(np.sum(lens))
    return B <= 192 and (total + (rows - 1) * B) // rows < B * ((int(np.max(lens)) + rows - 1) // rows)


@pytest.mark.parametrize("nseq", [192, 193])
def test_packed_many_sequences(nseq):
    """192 packed sequences (the most for which the grid holds only real
    tiles) and 193 (one CTA per sequence, head and tile of the longest, most
    of them empty), some of them empty: each sequence equals the oracle on
    its own slice."""
    H, d, dtype, wl, wr = 2, 128, sy.BF16, -1, 0
    rng = np.random.default_rng(9700 + nseq)
    lens = rng.integers(1, 300, nseq)
    lens[::17] = 0
    lens[7] = 300
    assert _tile_search_grid(lens) == (nseq <= 192)
    total = int(lens.sum())
    q, k, v = qkv(1, H, total, total, d, dtype, seed=9710 + nseq)
    qp, kp, vp = (np.ascontiguousarray(x[0].transpose(1, 0, 2)) for x in (q, k, v))   # [total, H, d]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    o, lse = fa2.fa2_fwd_ex(to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype), window_left=wl,
                            window_right=wr, cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=int(lens.max()))
    status_ok()
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    row = 0
    for i, n in enumerate(lens.tolist()):
        if n:
            sl = lambda x: np.ascontiguousarray(x[:, :, row:row + n])
            o_orc, l_orc = oracle.attention_fwd_masked(sl(q), sl(k), sl(v), dtype, 1.0 / np.sqrt(d),
                                                       window_left=wl, window_right=wr)
            og = o[row:row + n].transpose(1, 0, 2)[None]
            check(og, lse[None, :, row:row + n], o_orc, l_orc, dtype, "seq %d of %d (n=%d)" % (i, nseq, n))
        row += n


@pytest.mark.parametrize("trial", range(8))
def test_packed_random_mixes_bit_equal_unpacked(trial):
    """Random packed batches (1 to 200 sequences, skewed lengths with empty
    ones, N_q != N_k, any head count, head dim and mask): every sequence's
    rows bit-equal the unpacked call on that sequence alone, whichever grid
    the batch gets; rows outside every sequence stay untouched."""
    rng = np.random.default_rng(9800 + trial)
    nseq = int(rng.choice([1, 2, 7, 31, 64, 150, 192, 200]))
    d, dtype = [(64, sy.FP16), (128, sy.BF16), (256, sy.FP16), (128, sy.FP16)][trial % 4]
    H = int(rng.integers(1, 4))
    wl, wr, pre = [(-1, 0, 0), (-1, -1, 0), (int(rng.integers(0, 300)), 0, 0), (-1, 0, int(rng.integers(1, 200)))][trial % 4]
    scale_len = 2000 if nseq <= 31 else 400
    lq = np.minimum(rng.exponential(scale_len / 4, nseq).astype(np.int64), scale_len)
    lk = np.where(rng.random(nseq) < 0.5, lq, np.minimum(rng.exponential(scale_len / 4, nseq).astype(np.int64), scale_len))
    lq[rng.random(nseq) < 0.1] = 0
    lq[0] = max(int(lq[0]), 1)
    lk[0] = max(int(lk[0]), 1)
    tq, tk, tail = int(lq.sum()), int(lk.sum()), 5
    q, k, v = qkv(1, H, tq + tail, max(tk, 1), d, dtype, seed=9810 + trial)
    qp, kp, vp = (np.ascontiguousarray(x[0].transpose(1, 0, 2)) for x in (q, k, v))
    qd, kd, vd = to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32, device="cuda")
    mask = dict(window_left=wl, window_right=wr, prefix_len=pre)
    o = torch.full(qd.shape, 3.0, dtype=qd.dtype, device="cuda")
    lse = torch.full((H, qd.shape[0]), 4.0, dtype=torch.float32, device="cuda")
    fa2.fa2_fwd_ex(qd, kd, vd, o=o, lse=lse, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=int(lq.max()), **mask)
    status_ok()
    assert torch.all(o[tq:] == 3.0) and torch.all(lse[:, tq:] == 4.0)
    rq = rk = 0
    for i, (nq, nk) in enumerate(zip(lq.tolist(), lk.tolist())):
        if nq:
            og = o[rq:rq + nq].permute(1, 0, 2).unsqueeze(0)
            lg = lse[:, rq:rq + nq].unsqueeze(0)
            label = "trial %d seq %d of %d (nq=%d nk=%d) d=%d mask=%s" % (trial, i, nseq, nq, nk, d, (wl, wr, pre))
            if nk == 0:
                assert torch.all(og == 0) and torch.all(torch.isneginf(lg)), label
            else:
                ou, lu = _unpacked(qd, kd, vd, (rq, rq + nq), (rk, rk + nk), **mask)
                assert torch.equal(og, ou) and torch.equal(lg, lu), label + ": packed != unpacked"
        rq += nq
        rk += nk


def _unpacked(qd, kd, vd, q_rows, k_rows, **mask):
    sl = lambda x, r: x[r[0]:r[1]].permute(1, 0, 2).unsqueeze(0)
    o, lse = fa2.fa2_fwd_ex(sl(qd, q_rows), sl(kd, k_rows), sl(vd, k_rows), **mask)
    status_ok()
    return o, lse


def test_out_of_range_offsets_are_reported_and_skipped():
    """Offsets the kernel's own checks reject (keys decreasing, rows past
    total_q, more rows than max_seqlen_q): those sequences are left as they
    were, the others are written, and the status word reports
    FA2_ERR_DEVICE_SEQLENS."""
    H, d, dtype = 2, 128, sy.BF16
    q, k, v = qkv(1, H, 400, 400, d, dtype, seed=9400)
    qp, kp, vp = (np.ascontiguousarray(x[0].transpose(1, 0, 2)) for x in (q, k, v))   # [400, H, d]
    qd, kd, vd = to_dev(qp, dtype), to_dev(kp, dtype), to_dev(vp, dtype)
    causal = dict(window_left=-1, window_right=0)

    def call(cu_q, cu_k, max_q):
        o = torch.full(qd.shape, 3.0, dtype=qd.dtype, device="cuda")
        lse = torch.full((H, 400), 4.0, dtype=torch.float32, device="cuda")
        fa2.fa2_fwd_ex(qd, kd, vd, o=o, lse=lse, cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32, device="cuda"),
                       cu_seqlens_k=torch.tensor(cu_k, dtype=torch.int32, device="cuda"), max_seqlen_q=max_q, **causal)
        torch.cuda.synchronize()
        code, detail = fa2.fa2_get_device_status()
        assert code == fa2.FA2_ERR_DEVICE_SEQLENS, (code, hex(detail))
        return o.permute(1, 0, 2).unsqueeze(0), lse.unsqueeze(0)

    # seq 0 rows [0,100) keys [0,100); seq 1 no rows but keys decreasing (rejected);
    # seq 2 rows [100,300) keys [50,300); seq 3 rows [300,500) past total_q = 400 (rejected)
    o, lse = call([0, 100, 100, 300, 500], [0, 100, 50, 300, 400], 256)
    for rows, keys in (((0, 100), (0, 100)), ((100, 300), (50, 300))):
        ou, lu = _unpacked(qd, kd, vd, rows, keys, **causal)
        assert torch.equal(o[:, :, rows[0]:rows[1]], ou) and torch.equal(lse[:, :, rows[0]:rows[1]], lu)
    assert torch.all(o[:, :, 300:] == 3.0) and torch.all(lse[:, :, 300:] == 4.0)
    # seq 1 has 200 rows, more than max_seqlen_q = 150 (rejected); seq 0 still written
    o, lse = call([0, 100, 300], [0, 100, 300], 150)
    ou, lu = _unpacked(qd, kd, vd, (0, 100), (0, 100), **causal)
    assert torch.equal(o[:, :, :100], ou) and torch.equal(lse[:, :, :100], lu)
    assert torch.all(o[:, :, 100:] == 3.0) and torch.all(lse[:, :, 100:] == 4.0)


# ------------------------------------------------------------------ long sequences, sampled rows

@pytest.mark.parametrize("Nq,Nk,mask,d,dtype", [
    (16384, 16384, (4096, 0, 0), 128, sy.BF16),     # sliding window of 4096 keys
    (256, 16384, (-1, 0, 0), 128, sy.BF16),          # a 256-row chunk after a 16128-key prefix
    (8192, 8192, (-1, 0, 1024), 64, sy.FP16),       # prefix-LM with a 1024-key prefix
    (3000, 3000, (512, 512, 0), 256, sy.FP16),      # symmetric band
])
def test_long_sampled_rows(Nq, Nk, mask, d, dtype):
    wl, wr, pre = mask
    B, H = 1, 4
    q, k, v = qkv(B, H, Nq, Nk, d, dtype, seed=9500 + Nq)
    scale = 1.0 / np.sqrt(d)
    o, lse = run_ex(q, k, v, dtype, scale, window_left=wl, window_right=wr, prefix_len=pre)
    rng = np.random.default_rng(Nq)
    rows = np.unique(np.concatenate([np.arange(0, min(Nq, 3)), [Nq - 1, Nq // 2, min(Nq - 1, 128), min(Nq - 1, 255)],
                                     rng.integers(0, Nq, 24)]))
    bh = np.repeat(np.arange(B * H), rows.size)
    rr = np.tile(rows, B * H)
    o_ref, l_ref = oracle.attention_rows_masked(q, k, v, dtype, scale, bh, rr, window_left=wl, window_right=wr,
                                                prefix_len=pre)
    og = o.reshape(B * H, Nq, d)[bh, rr]
    lg = lse.reshape(B * H, Nq)[bh, rr]
    check(og, lg, o_ref, l_ref, dtype, "Nq=%d Nk=%d mask=%s" % (Nq, Nk, mask))


def test_repeated_calls_bit_identical():
    q, k, v = qkv(1, 8, 2000, 2500, 128, sy.BF16, seed=9600)
    qd, kd, vd = (to_dev(x, sy.BF16) for x in (q, k, v))
    first = fa2.fa2_fwd_ex(qd, kd, vd, window_left=300, window_right=0, prefix_len=17)
    for _ in range(3):
        again = fa2.fa2_fwd_ex(qd, kd, vd, window_left=300, window_right=0, prefix_len=17)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
    status_ok()
