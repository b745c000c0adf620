"""The seeded input generator: deterministic, N(0,1)-distributed, correctly rounded."""
import numpy as np
import pytest
import torch

from exact_tiled_attention_fa2_gb300 import synthetic as sy


def test_splitmix64_reference_values():
    # splitmix64 with state 0: the first outputs of the published generator
    out = sy.splitmix64(0, np.arange(3))
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_seed_sensitive():
    a = sy.make_qkv(1, 2, 33, 16, sy.BF16, 7)
    b = sy.make_qkv(1, 2, 33, 16, sy.BF16, 7)
    c = sy.make_qkv(1, 2, 33, 16, sy.BF16, 8)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    assert not np.array_equal(a[0], c[0])
    assert not np.array_equal(a[0], a[1]) and not np.array_equal(a[1], a[2])


def test_moments():
    x = sy.normals_f32(123, 0, 1 << 20).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs((x ** 4).mean() - 3.0) < 0.05


def test_rounding_matches_torch():
    x = sy.normals_f32(5, 0, 100000) * np.float32(7.0)
    np.testing.assert_array_equal(sy.f32_to_bits(x, sy.BF16),
                                  torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(sy.f32_to_bits(x, sy.FP16),
                                  torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(sy.bits_to_f32(sy.f32_to_bits(x, sy.BF16), sy.BF16),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_q_scale_only_touches_q():
    q1, k1, v1 = sy.make_qkv(1, 1, 8, 8, sy.FP16, 3)
    q3, k3, v3 = sy.make_qkv(1, 1, 8, 8, sy.FP16, 3, q_scale=3.0)
    np.testing.assert_array_equal(k1, k3)
    np.testing.assert_array_equal(v1, v3)
    raw = sy.normals_f32(3, 0, 64)
    np.testing.assert_array_equal(q3.reshape(-1), sy.f32_to_bits(raw * np.float32(3.0), sy.FP16))


@pytest.mark.parametrize("Nq,Nk,wl,wr,pre", [(7, 7, -1, -1, 0), (7, 7, -1, 0, 0), (5, 12, 2, 1, 0), (12, 5, -1, 0, 0),
                                             (20, 20, 3, 0, 4), (20, 20, 0, 0, 25), (9, 30, 0, -1, 2)])
def test_visible_keys_matches_brute_force(Nq, Nk, wl, wr, pre):
    off = Nk - Nq
    want = []
    for i in range(Nq):
        n = 0
        for j in range(Nk):
            band = (wl < 0 or j >= i + off - wl) and (wr < 0 or j <= i + off + wr)
            n += (j < pre) or band
        want.append(n)
    np.testing.assert_array_equal(sy.visible_keys(Nq, Nk, wl, wr, pre), want)


@pytest.mark.parametrize("Nq,Nk,wl,wr,pre", [(7, 7, -1, -1, 0), (7, 7, -1, 0, 0), (5, 12, 2, 1, 0), (12, 5, -1, 0, 0),
                                             (20, 20, 3, 0, 4), (20, 20, 0, 0, 25), (9, 30, 0, -1, 2),
                                             (1, 64, 4, 0, 0), (3, 100, 0, 0, 0), (8, 50, 10, 2, 30), (4, 4, 0, 0, 0)])
def test_union_visible_keys_matches_brute_force(Nq, Nk, wl, wr, pre):
    off = Nk - Nq
    seen = set()
    for i in range(Nq):
        for j in range(Nk):
            band = (wl < 0 or j >= i + off - wl) and (wr < 0 or j <= i + off + wr)
            if (j < pre) or band:
                seen.add(j)
    assert sy.union_visible_keys(Nq, Nk, wl, wr, pre) == len(seen)
