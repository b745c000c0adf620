"""Failure detection without a GPU fault: a kernel wait that can never be
satisfied gives up after its limit, records the wait site in the device
status word and returns; the host reads the timeout, the word is cleared and
the context stays usable for the next forward pass."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_fa2_gb300 as fa2
import oracle
from exact_tiled_attention_fa2_gb300 import build as fa2_build
from exact_tiled_attention_fa2_gb300 import synthetic as sy

pytestmark = pytest.mark.gpu

SITE_SELFTEST = 11


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa2_build.build()
    fa2.load_library()


def test_expired_wait_is_reported_and_cleared():
    code, _ = fa2.fa2_get_device_status()          # start from a clean word
    assert code == fa2.FA2_OK
    fa2.fa2_selftest_wait_timeout(2000)             # 2 ms limit on a wait nothing completes
    code, detail = fa2.fa2_get_device_status()
    assert code == fa2.FA2_ERR_DEVICE_TIMEOUT
    assert detail & 1 and detail & (1 << (8 + SITE_SELFTEST))
    code, detail = fa2.fa2_get_device_status()      # reading cleared it
    assert code == fa2.FA2_OK and detail == 0


def test_context_usable_after_expired_wait():
    fa2.fa2_selftest_wait_timeout(1000)
    assert fa2.fa2_get_device_status()[0] == fa2.FA2_ERR_DEVICE_TIMEOUT
    q, k, v = sy.make_qkv(1, 2, 200, 128, sy.BF16, 8101)
    dev = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in (q, k, v)]
    o, lse = fa2.fa2_fwd(*dev, causal=True)
    torch.cuda.synchronize()
    assert fa2.fa2_get_device_status()[0] == fa2.FA2_OK
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, sy.BF16, 1 / np.sqrt(128), True)
    assert np.abs(o.double().cpu().numpy() - o_ref).max() <= 1e-2
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3
