"""The core backward entry point that allocates nothing.

upipe_attn_core_bwd_noalloc is for callers that may not allocate device
memory at the point of the call (for example a framework's allocator during
its own out-of-memory handling, or a runtime with a fixed, fully claimed
memory budget).  Its scratch is a fixed array in the library's static device
memory.  These checks call it through the C ABI twice in a row (the array
keeps the previous call's contents) and compare with the workspace entry
point upipe_attn_core_bwd, within the parity tolerance and bit for bit.

This file is collected last on purpose: a run that stops at the first
failure has then already run every other test.
"""

import ctypes

import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from tests.gpu_common import dev, ensure_lib, f64, status_ok
from tests.tolerance import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("L,H,Hkv,U", [(1000, 4, 1, 1), (2048, 8, 2, 4), (129, 4, 2, 2)])
def test_noalloc_core_backward_matches_workspace_entry(L, H, Hkv, U):
    ensure_lib()
    cfg = upipe.Config(L=L, H=H, Hkv=Hkv, U=U)
    assert upipe.workspace_bytes(cfg, 1, core_only=True) <= upipe.NOALLOC_SCRATCH_BYTES
    q, k, v, do = dev(*synth.core_inputs(L, H, Hkv))
    o, lse = upipe.core_forward(cfg, q, k, v)
    ref = upipe.core_backward(cfg, q, k, v, o, lse, do)
    torch.cuda.synchronize()
    for call in range(2):
        outs = [torch.full_like(t, float("nan")) for t in ref]
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info()[0]
        upipe.attn_core_bwd_noalloc(cfg, q, k, v, o, lse, do, *outs)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        if call == 1:
            # The first call may create the library's second stream; after
            # it, the device's free memory (which also sees allocations made
            # inside the library, outside torch's allocator) must not move.
            assert torch.cuda.mem_get_info()[0] == free_before, "the call allocated device memory"
        status_ok()
        for name, got, want in zip(("dq", "dk", "dv"), outs, ref):
            assert_close(f64(got), f64(want), f"{name} (call {call})")
            assert torch.equal(got, want), f"{name} (call {call}) differs from the workspace entry point"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = ensure_lib()
    # U = 1 with Hkv = 1 carries dK/dV in fp32: ~1 KiB of scratch per token.
    cfg = upipe.Config(L=1 << 20, H=4, Hkv=1, U=1).c()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected before any GPU work
    rc = lib.upipe_attn_core_bwd_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                         None)
    assert rc == upipe.UPIPE_ERR_SCRATCH_LIMIT
    assert "scratch" in upipe.strerror(rc)
