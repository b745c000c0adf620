"""fa2_fwd_host_noalloc: the host-buffer entry point for callers that cannot
allocate device memory (their device memory is reserved by another allocator,
or they must not call an allocator that may synchronise the device).  It
stages q, k, v, o and lse in the library's static device array instead of a
caller-provided workspace, so its results must equal those of fa2_fwd_host.

Collected last on purpose (file name), and independent of every other test:
it builds and loads the library itself.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu

TOL_O = {sy.FP16: 2e-3, sy.BF16: 1e-2}
TOL_LSE = 1e-3
TORCH_DT = {sy.FP16: torch.float16, sy.BF16: torch.bfloat16}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa2_build.build()
    return fa2.load_library()


def _host(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype]).pin_memory()


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    # two different problems back to back: the second call must not see the first one's data
    cases = [(1, 4, 1000, 128, sy.BF16, True, 9101), (2, 3, 777, 64, sy.FP16, False, 9102)]
    for B, H, N, d, dtype, causal, seed in cases:
        assert fa2.fa2_fwd_host_workspace_bytes(B, H, N, d) <= fa2.FA2_NOALLOC_SCRATCH_BYTES
        q, k, v = (_host(x, dtype) for x in sy.make_qkv(B, H, N, d, dtype, seed))
        scale = 1.0 / np.sqrt(d)
        o_a = torch.empty((B, H, N, d), dtype=TORCH_DT[dtype]).pin_memory()
        l_a = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        stream = torch.cuda.current_stream()
        rc = lib.fa2_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_a.data_ptr(), l_a.data_ptr(),
                                      B, H, N, d, ctypes.c_float(scale), int(causal), dtype,
                                      ctypes.c_void_p(stream.cuda_stream))
        assert rc == fa2.FA2_OK, fa2.fa2_status_string(rc)
        o_b = torch.empty_like(o_a).pin_memory()
        l_b = torch.empty_like(l_a).pin_memory()
        ws = torch.empty(fa2.fa2_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
        fa2.fa2_fwd_host(q, k, v, o_b, l_b, ws, scale=scale, causal=causal)
        assert torch.isfinite(o_a.float()).all() and torch.isfinite(l_a).all()
        assert (o_a.double() - o_b.double()).abs().max().item() <= TOL_O[dtype]
        assert (l_a.double() - l_b.double()).abs().max().item() <= TOL_LSE


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    tiny = torch.zeros(16, dtype=torch.float16).pin_memory()
    lse = torch.zeros(16, dtype=torch.float32).pin_memory()
    B, H, N, d = 1, 16, 4096, 128   # needs 64 MiB + 256 KiB of staging
    assert fa2.fa2_fwd_host_workspace_bytes(B, H, N, d) > fa2.FA2_NOALLOC_SCRATCH_BYTES
    # rejected on size before any copy, so the small buffers are never touched
    rc = lib.fa2_fwd_host_noalloc(tiny.data_ptr(), tiny.data_ptr(), tiny.data_ptr(), tiny.data_ptr(), lse.data_ptr(),
                                  B, H, N, d, ctypes.c_float(0.088), 1, sy.FP16, None)
    assert rc == fa2.FA2_ERR_SCRATCH_LIMIT
    assert "static device scratch" in fa2.fa2_status_string(rc)
