"""Failure detection without a GPU fault.

Every wait in the library's kernels is bounded; when one expires the kernel
records a timeout in the device status word and returns.  A diagnostics
kernel waits on a barrier that nothing arrives at, so its wait must expire:
the host must then read PATH_ERR_TIMEOUT, the word must clear, and the
context must stay usable for a normal forward call.
"""
import numpy as np
import pytest
import torch

import householder_softmax_attention_gb300 as pa
from seeded_inputs import Workload, make_inputs

PATH_ERR_TIMEOUT = -4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from householder_softmax_attention_gb300 import build
    build.build()
    pa.load_library()


@pytest.mark.gpu
def test_expired_wait_is_reported_and_context_survives():
    assert pa.path_attn_device_status(0, True) == 0
    pa.path_attn_debug_wait_timeout(20_000_000)  # 20 ms
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, True) == PATH_ERR_TIMEOUT
    assert pa.path_attn_device_status(0, True) == 0  # cleared
    wl = Workload("after_timeout", 1, 2, 300, 64, "bf16", seed=77)
    x = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in make_inputs(wl).items()}
    o1, l1 = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, x["scale"])
    o2, l2 = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], None, x["scale"])
    torch.cuda.synchronize()
    assert pa.path_attn_device_status(0, True) == 0
    assert torch.isfinite(o1.float()).all() and torch.equal(o1, o2)


def test_wait_limit_is_validated_on_the_host():
    lib = pa.load_library()
    assert lib.path_attn_debug_wait_timeout(0, None) == -1
    assert lib.path_attn_debug_wait_timeout(10**12, None) == -1
