"""Activation offload through the C ABI (GPU): the layer's block input x is
copied to pinned host memory after the forward, removed from the device,
prefetched back before the backward, and the backward returns the same bits
as with x resident; copies in both directions run beside the layer's
kernels without changing their results."""

import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from tests.gpu_common import ensure_lib, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _layer(shape):
    cfg = upipe.Config(L=shape.L, D=shape.D, H=shape.H, Hkv=shape.Hkv, U=shape.U, rope_theta=shape.theta)
    return cfg, [t.to("cuda:0") for t in synth.layer_inputs(shape)]


def test_offloaded_and_prefetched_input_gives_identical_gradients():
    shape = synth.LayerShape(L=4096, D=1024, H=8, Hkv=2, U=2)
    cfg, (x, w, wo, dout) = _layer(shape)
    out, lse, _ = upipe.layer_forward(cfg, x, w, wo)
    ref = upipe.layer_backward(cfg, x, w, wo, dout, lse)
    torch.cuda.synchronize()
    host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_copy = x.clone()
    upipe.offload_async(host, x)
    upipe.copies_join()
    x.fill_(float("nan"))  # the device copy is gone (overwritten after the join)
    torch.cuda.synchronize()
    assert torch.equal(host, x_copy.cpu())
    upipe.prefetch_async(x, host)
    upipe.copies_join()
    got = upipe.layer_backward(cfg, x, w, wo, dout, lse)
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(x, x_copy)
    for a, b, n in zip(got, ref, ("dx", "dWqkv", "dWo")):
        assert torch.equal(a, b), f"{n} differs after the round trip through host memory"


def test_copies_in_flight_beside_the_layer_change_nothing():
    """An offload and a prefetch of 256 MiB each run on the copy streams while
    the layer computes on the caller's stream; the layer's results equal the
    undisturbed run, and both copies arrive intact."""
    shape = synth.LayerShape(L=8192, D=2048, H=16, Hkv=4, U=4)
    cfg, (x, w, wo, dout) = _layer(shape)
    out0, lse0, _ = upipe.layer_forward(cfg, x, w, wo)
    ref = upipe.layer_backward(cfg, x, w, wo, dout, lse0)
    torch.cuda.synchronize()
    n = 128 << 20  # bf16 elements: 256 MiB each way
    src_dev = torch.randn(n, device="cuda:0").to(torch.bfloat16)
    dst_host = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    src_host = torch.randn(n).to(torch.bfloat16).pin_memory()
    dst_dev = torch.empty(n, dtype=torch.bfloat16, device="cuda:0")
    torch.cuda.synchronize()
    upipe.offload_async(dst_host, src_dev)
    upipe.prefetch_async(dst_dev, src_host)
    out, lse, _ = upipe.layer_forward(cfg, x, w, wo)
    got = upipe.layer_backward(cfg, x, w, wo, dout, lse)
    upipe.copies_join()
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(out, out0) and torch.equal(lse, lse0)
    for a, b, name in zip(got, ref, ("dx", "dWqkv", "dWo")):
        assert torch.equal(a, b), name
    assert torch.equal(dst_host, src_dev.cpu())
    assert torch.equal(dst_dev.cpu(), src_host)


def test_offload_rejects_bad_arguments():
    dev_t = torch.zeros(16, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(ValueError):
        upipe.offload_async(torch.zeros(8, dtype=torch.bfloat16), dev_t)
    with pytest.raises(ValueError):
        upipe.prefetch_async(dev_t, torch.zeros(16, dtype=torch.float32))
    lib = upipe.lib()
    assert lib.upipe_offload_async(None, None, 0, None) == upipe.UPIPE_OK
    assert lib.upipe_offload_async(None, None, 16, None) == upipe.UPIPE_ERR_INVALID_ARG
