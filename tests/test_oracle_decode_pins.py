"""Pins for the split-over-keys (decoding) restatement: for few query rows and
many keys, per-chunk online-softmax states merged by the rescaling step equal
the plain definition (the pinned masked oracle) for every chunking and mask;
chunks that show a row nothing are handled; merging without the rescaling
factors breaks it.  CPU only."""
import numpy as np
import pytest

import oracle
from exact_tiled_attention_fa2_gb300 import synthetic as sy
from oracle.tiled_reference import split_keys_attention


def _visible(nq, nk, wl, wr, pre):
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    off = nk - nq
    band = np.ones((nq, nk), dtype=bool)
    if wl >= 0:
        band &= j >= i + off - wl
    if wr >= 0:
        band &= j <= i + off + wr
    return band | (j < pre)


MASKS = [(-1, -1, 0), (-1, 0, 0), (40, 0, 0), (-1, 0, 17), (3, 2, 0)]


@pytest.mark.parametrize("chunk", [1, 7, 64, 333, 1000])
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("nq", [1, 4])
def test_split_keys_equals_the_definition(chunk, mask, nq):
    nk, d = 333, 16
    dtype = sy.BF16
    q = sy.make_qkv(1, 2, nq, d, dtype, 31)[0]
    _, k, v = sy.make_qkv(1, 2, nk, d, dtype, 32)
    wl, wr, pre = mask
    o_ref, l_ref = oracle.attention_fwd_masked(q, k, v, dtype, 0.4, window_left=wl, window_right=wr, prefix_len=pre)
    Q, K, V = (oracle.widen(x, dtype) for x in (q, k, v))
    vis = _visible(nq, nk, wl, wr, pre)
    for h in range(2):
        o, l = split_keys_attention(Q[0, h], K[0, h], V[0, h], 0.4, chunk, vis)
        np.testing.assert_allclose(o, o_ref[0, h], atol=1e-13, rtol=0)
        np.testing.assert_allclose(l, l_ref[0, h], atol=1e-12, rtol=0)


def test_chunks_showing_nothing_and_rows_without_keys():
    # window (3, 0) near the end of 300 keys: every chunk but the last shows the rows nothing;
    # N_q > N_k under causal leaves the first rows without any key at all
    q = sy.make_qkv(1, 1, 6, 8, sy.FP16, 41)[0]
    _, k, v = sy.make_qkv(1, 1, 300, 8, sy.FP16, 42)
    Q, K, V = (oracle.widen(x, sy.FP16)[0, 0] for x in (q, k, v))
    o, l = split_keys_attention(Q, K, V, 1.0, 64, _visible(6, 300, 3, 0, 0))
    o_ref, l_ref = oracle.attention_fwd_masked(q, k, v, sy.FP16, 1.0, window_left=3, window_right=0)
    np.testing.assert_allclose(o, o_ref[0, 0], atol=1e-13, rtol=0)
    np.testing.assert_allclose(l, l_ref[0, 0], atol=1e-12, rtol=0)
    q = sy.make_qkv(1, 1, 10, 8, sy.FP16, 43)[0]
    _, k, v = sy.make_qkv(1, 1, 4, 8, sy.FP16, 44)
    Q, K, V = (oracle.widen(x, sy.FP16)[0, 0] for x in (q, k, v))
    o, l = split_keys_attention(Q, K, V, 1.0, 2, _visible(10, 4, -1, 0, 0))
    assert np.all(o[:6] == 0) and np.all(np.isneginf(l[:6])) and np.isfinite(l[6:]).all()


def test_merging_without_rescaling_is_not_exact():
    q = sy.make_qkv(1, 1, 2, 16, sy.FP16, 51, q_scale=3.0)[0]
    _, k, v = sy.make_qkv(1, 1, 256, 16, sy.FP16, 52)
    Q, K, V = (oracle.widen(x, sy.FP16)[0, 0] for x in (q, k, v))
    good, _ = split_keys_attention(Q, K, V, 0.5, 32)
    bad, _ = split_keys_attention(Q, K, V, 0.5, 32, merge_rescale=False)
    assert np.abs(good - bad).max() > 1e-2
