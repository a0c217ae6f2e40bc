"""The autograd front end (headwise_chunked_context_gb300/modules.py) returns
the library's own results: module forward and parameter / input gradients
equal the binding's calls bit for bit, and a block of the three modules
trains (one SGD step lowers the loss)."""

import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from headwise_chunked_context_gb300.modules import HeadChunkedAttention, TiledCrossEntropy, TiledSwiGLU
from tests.gpu_common import ensure_lib, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


@pytest.mark.parametrize("keep", [None, "device_o", "host"])
def test_attention_module_equals_the_binding(keep):
    torch.manual_seed(0)
    L, D, H, Hkv, U = 640, 256, 8, 2, 2
    m = HeadChunkedAttention(D, H, Hkv, U, keep=keep)
    x = torch.randn(L, D, device="cuda").bfloat16().requires_grad_()
    dout = torch.randn(L, D, device="cuda").bfloat16()
    out = m(x)
    out.backward(dout)
    torch.cuda.synchronize()
    status_ok()
    cfg = upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=U)
    wq, wo = m.wqkv.detach().bfloat16(), m.wo.detach().bfloat16()
    kmap = {None: False, "device_o": True, "host": "host"}
    r_out, lse, kept = upipe.layer_forward(cfg, x.detach(), wq, wo, keep_o=kmap[keep])
    r_dx, r_dw, r_dwo = upipe.layer_backward(cfg, x.detach(), wq, wo, dout, lse, kept)
    assert torch.equal(out, r_out) and torch.equal(x.grad, r_dx)
    assert torch.equal(m.wqkv.grad, r_dw) and torch.equal(m.wo.grad, r_dwo)


def test_mlp_and_loss_modules_equal_the_binding():
    torch.manual_seed(1)
    L, D, F, V, T = 300, 256, 384, 1024, 128
    mlp, ce = TiledSwiGLU(D, F, T), TiledCrossEntropy(D, V, T)
    x = torch.randn(L, D, device="cuda").bfloat16().requires_grad_()
    _, _, labels = synth.ce_inputs(L, D, V, device="cuda")
    y = mlp(x)
    loss = ce(y, labels)
    loss.backward()
    torch.cuda.synchronize()
    status_ok()
    wgu, wd, w = mlp.wgu.detach().bfloat16(), mlp.wd.detach().bfloat16(), ce.w.detach().bfloat16()
    r_y = upipe.mlp_forward(x.detach(), wgu, wd, T)
    scale = 1.0 / int((labels >= 0).sum())
    r_loss, r_dh, r_dw = upipe.ce_loss(r_y, w, labels, scale, T)
    r_dx, r_dwgu, r_dwd = upipe.mlp_backward(x.detach(), wgu, wd, r_dh, T)
    assert torch.equal(y, r_y)
    assert torch.allclose(loss, r_loss.sum() * scale, rtol=0, atol=0)
    assert torch.equal(ce.w.grad, r_dw) and torch.equal(x.grad, r_dx)
    assert torch.equal(mlp.wgu.grad, r_dwgu) and torch.equal(mlp.wd.grad, r_dwd)


def test_a_block_of_the_three_modules_trains():
    torch.manual_seed(2)
    L, D, H, Hkv, U, F, V = 512, 256, 4, 2, 2, 512, 512
    attn, mlp, ce = HeadChunkedAttention(D, H, Hkv, U), TiledSwiGLU(D, F, 256), TiledCrossEntropy(D, V, 256)
    params = [*attn.parameters(), *mlp.parameters(), *ce.parameters()]
    x = torch.randn(L, D, device="cuda").bfloat16()
    labels = torch.randint(0, V, (L,), device="cuda", dtype=torch.int32)
    opt = torch.optim.SGD(params, lr=0.5)
    losses = []
    for _ in range(3):
        opt.zero_grad()
        h = attn(x)
        loss = ce(mlp(h) + h, labels)
        loss.backward()
        losses.append(float(loss.detach()))
        assert all(torch.isfinite(p.grad).all() for p in params)
        opt.step()
    status_ok()
    assert losses[-1] < losses[0]
