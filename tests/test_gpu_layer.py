"""GPU parity of the whole head-chunked layer (projections, RoPE, causal
attention, output projection; forward and backward) against the fp64
oracle, through the C ABI, and bit-exactness of every chunk size against
the unchunked run (U = H).

The bound applies against the oracle's precision-model mode ("bf16 in /
fp32 accumulate": every contraction input -- Q, K, V, O, dO and the softmax
tiles P and dS where they enter a product -- rounded to bf16, everything
else exact fp64).  Each result is also compared with the plain fp64
definition, bounded by the stated rel-L2 and, for max-abs, by the precision
model's own deviation plus the tolerance (tests/tolerance.py)."""

import numpy as np
import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from oracle import upipe_oracle as orc
from tests.gpu_common import dev, ensure_lib, f64, status_ok
from tests.tolerance import assert_close, assert_close_plain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _run(shape, U, keep_o=False):
    x, wqkv, wo, dout = synth.layer_inputs(shape)
    cfg = upipe.Config(L=shape.L, D=shape.D, H=shape.H, Hkv=shape.Hkv, U=U, rope_theta=shape.theta)
    xd, wd, wod, dd = dev(x, wqkv, wo, dout)
    out, lse, o_saved = upipe.layer_forward(cfg, xd, wd, wod, keep_o=keep_o)
    dx, dwqkv, dwo = upipe.layer_backward(cfg, xd, wd, wod, dd, lse, o_saved)
    torch.cuda.synchronize()
    status_ok()
    return (x, wqkv, wo, dout), (out, lse, dx, dwqkv, dwo)


def _check_vs_oracle(shape, inputs, outs, kept_o=False):
    x, wqkv, wo, dout = (f64(t) for t in inputs)
    got = [f64(t) for t in outs]
    names = ("out", "lse", "dx", "dWqkv", "dWo")
    wgrad = (False, False, False, True, True)
    args = (x, wqkv, wo, shape.H, shape.Hkv, shape.theta)
    m_out, m_lse, _ = orc.layer_fwd(*args, bf16_operands=True)
    m_bwd = orc.layer_bwd(x, wqkv, wo, dout, shape.H, shape.Hkv, shape.theta, bf16_operands=True, kept_o=kept_o)
    model = (m_out, m_lse, *m_bwd)
    for g_, m, n, wg in zip(got, model, names, wgrad):
        assert_close(g_, m, n, weight_grad=wg)
    p_out, p_lse, _ = orc.layer_fwd(*args)
    p_bwd = orc.layer_bwd(x, wqkv, wo, dout, shape.H, shape.Hkv, shape.theta)
    for g_, p, m, n, wg in zip(got, (p_out, p_lse, *p_bwd), model, names, wgrad):
        assert_close_plain(g_, p, m, n, weight_grad=wg)


def test_tiny_config_matches_oracle():
    """L=1024, D=1024, H=8, Hkv=2, U=2 (U < g), theta=500000."""
    inputs, outs = _run(synth.TINY, synth.TINY.U)
    _check_vs_oracle(synth.TINY, inputs, outs)


# L = 1 and 64: one K block in the weight-gradient GEMM (no K split); 65: two
# blocks, the second holding one token.
@pytest.mark.parametrize("L,D,H,Hkv,U", [(200, 256, 4, 2, 2), (129, 128, 4, 1, 1), (384, 384, 8, 2, 4),
                                         (1, 128, 2, 1, 1), (64, 256, 4, 2, 2), (65, 256, 4, 2, 2)])
def test_ragged_layers_match_oracle(L, D, H, Hkv, U):
    shape = synth.LayerShape(L=L, D=D, H=H, Hkv=Hkv, U=U)
    inputs, outs = _run(shape, U)
    _check_vs_oracle(shape, inputs, outs)


@pytest.mark.parametrize("L,D,H,Hkv", [(1024, 1024, 8, 2), (333, 256, 8, 4)])
def test_every_chunk_size_is_bit_exact_to_unchunked(L, D, H, Hkv):
    shape = synth.LayerShape(L=L, D=D, H=H, Hkv=Hkv)
    g = H // Hkv
    _, ref = _run(shape, H)
    for U in [u for u in range(1, H) if H % u == 0 and (u % g == 0 or g % u == 0)]:
        _, outs = _run(shape, U)
        for a, b, n in zip(ref, outs, ("out", "lse", "dx", "dWqkv", "dWo")):
            assert torch.equal(a, b), f"U={U}: {n} differs from the unchunked run"


def test_saved_o_matches_recompute():
    """A kept O and a recomputed O are both written from the final softmax
    probabilities, so the backward returns identical bits either way; the
    forward's `out` without a kept O comes from the online softmax and
    agrees within the tolerance."""
    shape = synth.LayerShape(L=300, D=256, H=4, Hkv=2)
    inputs, a = _run(shape, 2, keep_o=False)
    _, b = _run(shape, 2, keep_o=True)
    for x, y, n in list(zip(a, b, ("out", "lse", "dx", "dWqkv", "dWo")))[1:]:
        assert torch.equal(x, y), n
    assert_close(f64(a[0]), f64(b[0]), "out (online softmax) vs out (kept O)")
    _check_vs_oracle(shape, inputs, b)


@pytest.mark.parametrize("L,D,H,Hkv,U", [(1024, 1024, 8, 2, 2), (300, 256, 4, 2, 4), (129, 128, 4, 1, 1),
                                         (65, 256, 8, 2, 1)])
def test_host_o_matches_oracle(L, D, H, Hkv, U):
    """O kept in page-locked host memory (one and several chunks; with four
    and more chunks both staging buffers are reused).  The forward is the
    recomputing forward's bit for bit; the backward reads the forward's own
    O, which the oracle's kept-O model describes (the two backward modes
    differ by the bf16 rounding of two different O, the precision model's
    own deviation, so each is checked against its own model)."""
    shape = synth.LayerShape(L=L, D=D, H=H, Hkv=Hkv, U=U)
    inputs, h = _run(shape, U, keep_o="host")
    _, r = _run(shape, U)
    assert torch.equal(h[0], r[0]) and torch.equal(h[1], r[1]), "forward differs from the recomputing forward"
    _check_vs_oracle(shape, inputs, h, kept_o=True)


def test_host_o_every_chunk_size_is_bit_exact_to_unchunked():
    shape = synth.LayerShape(L=333, D=256, H=8, Hkv=4)
    _, ref = _run(shape, 8, keep_o="host")
    for U in (1, 2, 4):
        _, outs = _run(shape, U, keep_o="host")
        for a, b, n in zip(ref, outs, ("out", "lse", "dx", "dWqkv", "dWo")):
            assert torch.equal(a, b), f"U={U}: {n} differs from the unchunked run"
