"""Bounded device waits: a wait on an mbarrier that nothing arrives on runs
out, sets the status word, and leaves the context usable."""

import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from tests.gpu_common import dev, ensure_lib

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_status_and_context_survives():
    ensure_lib()
    assert upipe.last_device_status() == 0
    upipe.debug_wait_timeout(2_000_000)  # 2 ms
    assert upipe.last_device_status() == upipe.UPIPE_ERR_DEVICE_TIMEOUT
    assert upipe.last_device_status() == 0  # reading clears it
    q, k, v, _ = synth.core_inputs(256, 2, 1)
    cfg = upipe.Config(L=256, H=2, Hkv=1, U=1)
    o, lse = upipe.core_forward(cfg, *dev(q, k, v))
    torch.cuda.synchronize()
    assert upipe.last_device_status() == 0
    assert torch.isfinite(o.float()).all()
