"""fa2_fwd_host_noalloc: the host-buffer entry point for callers that cannot
allocate device memory (their device memory is reserved by another allocator,
or they must not call an allocator that may synchronise the device).  It
stages q, k, v, o and lse in the library's static device array instead of a
caller-provided workspace and runs the same kernel on the same inputs, so its
results must equal fa2_fwd_host's bit for bit.

Collected last on purpose (file name), and independent of every other test:
it builds and loads the library itself.
"""
import ctypes

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


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa2_build.build()
    return fa2.load_library()


def _host(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH_DT[dtype]).pin_memory()


def _noalloc(lib, q, k, v, B, H, N, d, dtype, causal):
    o = torch.empty((B, H, N, d), dtype=TORCH_DT[dtype]).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()
    rc = lib.fa2_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  B, H, N, d, ctypes.c_float(1.0 / np.sqrt(d)), int(causal), dtype,
                                  ctypes.c_void_p(stream.cuda_stream))
    assert rc == fa2.FA2_OK, fa2.fa2_status_string(rc)
    return o, lse


def _with_workspace(q, k, v, B, H, N, d, dtype, causal):
    o = torch.empty((B, H, N, d), dtype=TORCH_DT[dtype]).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa2.fa2_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa2.fa2_fwd_host(q, k, v, o, lse, ws, scale=1.0 / np.sqrt(d), causal=causal)
    return o, lse


def _check_oracle(o, lse, bits, B, H, N, d, dtype, causal):
    o_ref, lse_ref = oracle.attention_fwd(*bits, dtype, 1.0 / np.sqrt(d), causal)
    eo = float(np.abs(o.double().numpy() - o_ref).max())
    el = float(np.abs(lse.double().numpy() - lse_ref).max())
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, (eo, el)


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    # call 1: a causal bf16 problem
    B, H, N, d, dtype, causal = 1, 4, 1000, 128, sy.BF16, True
    assert fa2.fa2_fwd_host_workspace_bytes(B, H, N, d) <= fa2.FA2_NOALLOC_SCRATCH_BYTES
    bits = sy.make_qkv(B, H, N, d, dtype, 9101)
    q, k, v = (_host(x, dtype) for x in bits)
    o_a, l_a = _noalloc(lib, q, k, v, B, H, N, d, dtype, causal)
    o_b, l_b = _with_workspace(q, k, v, B, H, N, d, dtype, causal)
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
    _check_oracle(o_a, l_a, bits, B, H, N, d, dtype, causal)

    # the array keeps the last call's contents: fill every byte call 2 will use
    # with NaN through a problem at least as large whose inputs are all NaN
    nan = torch.full((B, H, N, d), float("nan"), dtype=TORCH_DT[dtype]).pin_memory()
    _noalloc(lib, nan, nan, nan, B, H, N, d, dtype, False)

    # call 2: a smaller fp16 problem must see none of that: finite, equal to the
    # workspace entry point, and within the tolerances of the oracle
    B, H, N, d, dtype, causal = 2, 3, 777, 64, sy.FP16, False
    assert fa2.fa2_fwd_host_workspace_bytes(B, H, N, d) <= fa2.fa2_fwd_host_workspace_bytes(1, 4, 1000, 128)
    bits = sy.make_qkv(B, H, N, d, dtype, 9102)
    q, k, v = (_host(x, dtype) for x in bits)
    o_a, l_a = _noalloc(lib, q, k, v, B, H, N, d, dtype, causal)
    assert torch.isfinite(o_a.float()).all() and torch.isfinite(l_a).all()
    o_b, l_b = _with_workspace(q, k, v, B, H, N, d, dtype, causal)
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
    _check_oracle(o_a, l_a, bits, B, H, N, d, dtype, causal)


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
