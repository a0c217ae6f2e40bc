"""Pins of the sequence-tiled MLP / loss oracle (oracle/alst_oracle.py)
against things other than itself: torch float64 autograd and
``cross_entropy``, closed forms (silu at 0, uniform logits), invariants
(softmax-gradient rows sum to zero, tiled equals untiled) and finite
differences."""

import math

import numpy as np
import pytest
import torch

from oracle import alst_oracle as alst
from oracle.upipe_oracle import bf16_round


def _mlp_inputs(seed=0, L=40, D=24, F=16):
    r = np.random.default_rng(seed)
    x = r.standard_normal((L, D))
    Wgu = 0.3 * r.standard_normal((2 * F, D))
    Wd = 0.3 * r.standard_normal((D, F))
    dy = r.standard_normal((L, D))
    return x, Wgu, Wd, dy


def _ce_inputs(seed=0, L=33, D=16, V=40):
    r = np.random.default_rng(seed)
    h = r.standard_normal((L, D))
    W = 0.5 * r.standard_normal((V, D))
    labels = r.integers(0, V, L)
    labels[[3, 17, 30]] = -1  # ignored tokens
    return h, W, labels


def test_mlp_matches_torch_autograd():
    x, Wgu, Wd, dy = _mlp_inputs()
    F = Wd.shape[1]
    tx, tgu, td = (torch.tensor(a, requires_grad=True) for a in (x, Wgu, Wd))
    gu = tx @ tgu.T
    y = (torch.nn.functional.silu(gu[:, :F]) * gu[:, F:]) @ td.T
    (y * torch.tensor(dy)).sum().backward()
    ry, _ = alst.mlp_fwd(x, Wgu, Wd)
    dx, dWgu, dWd = alst.mlp_bwd(x, Wgu, Wd, dy)
    np.testing.assert_allclose(ry, y.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dx, tx.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dWgu, tgu.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dWd, td.grad.numpy(), atol=1e-12)


def test_mlp_backward_matches_finite_differences():
    x, Wgu, Wd, dy = _mlp_inputs(seed=1, L=6, D=5, F=4)
    dx, dWgu, dWd = alst.mlp_bwd(x, Wgu, Wd, dy)
    f = lambda x_, a_, b_: float(np.sum(alst.mlp_fwd(x_, a_, b_)[0] * dy))
    r = np.random.default_rng(9)
    eps = 1e-6
    for arg, grad in ((0, dx), (1, dWgu), (2, dWd)):
        args = [x, Wgu, Wd]
        v = r.standard_normal(args[arg].shape)
        plus = list(args)
        minus = list(args)
        plus[arg] = args[arg] + eps * v
        minus[arg] = args[arg] - eps * v
        fd = (f(*plus) - f(*minus)) / (2 * eps)
        assert abs(fd - float(np.sum(grad * v))) < 1e-7 * max(1.0, abs(fd))


def test_mlp_closed_form_at_zero_gate():
    """With Wg = 0 every gate is 0: silu(0) = 0 so H = 0, y = 0 and dWd = 0,
    silu'(0) = 1/2 so dG = dH * u / 2, and dU = dH * silu(0) = 0."""
    x, Wgu, Wd, dy = _mlp_inputs(seed=2)
    F = Wd.shape[1]
    Wgu[:F] = 0.0
    y, h = alst.mlp_fwd(x, Wgu, Wd)
    assert np.all(h == 0) and np.all(y == 0)
    dx, dWgu, dWd = alst.mlp_bwd(x, Wgu, Wd, dy)
    assert np.all(dWd == 0)
    u = x @ Wgu[F:].T
    dg = (dy @ Wd) * u * 0.5
    np.testing.assert_allclose(dWgu[:F], dg.T @ x, atol=1e-12)
    assert np.all(dWgu[F:] == 0)
    np.testing.assert_allclose(dx, dg @ Wgu[:F], atol=1e-12)


def test_ce_matches_torch_cross_entropy_and_autograd():
    h, W, labels = _ce_inputs()
    scale = 1.0 / np.count_nonzero(labels >= 0)
    th, tw = torch.tensor(h, requires_grad=True), torch.tensor(W, requires_grad=True)
    tl = torch.tensor(np.where(labels >= 0, labels, -100))
    loss_t = torch.nn.functional.cross_entropy(th @ tw.T, tl, reduction="none", ignore_index=-100)
    (scale * loss_t.sum()).backward()
    loss, dh, dW = alst.ce_fwd_bwd(h, W, labels, scale)
    np.testing.assert_allclose(loss, loss_t.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dh, th.grad.numpy(), atol=1e-13)
    np.testing.assert_allclose(dW, tw.grad.numpy(), atol=1e-13)


def test_ce_closed_forms():
    """Uniform logits (W = 0): every valid token's loss is log V and its
    logit gradient is scale (1/V - onehot); every row of the logit gradient
    sums to zero, so dh and dW are those of that dz."""
    h, W, labels = _ce_inputs(seed=3)
    V = W.shape[0]
    loss, dh, dW = alst.ce_fwd_bwd(h, np.zeros_like(W), labels, 0.5)
    valid = labels >= 0
    np.testing.assert_allclose(loss[valid], math.log(V), atol=1e-14)
    assert np.all(loss[~valid] == 0) and np.all(dh == 0)  # dh = dz W = 0
    dz = np.where(valid[:, None], np.full((len(labels), V), 0.5 / V), 0.0)
    dz[np.arange(len(labels))[valid], labels[valid]] -= 0.5
    np.testing.assert_allclose(dW, dz.T @ h, atol=1e-14)
    # Shifting every vocabulary row of W by one vector c adds h_i . c to all
    # of row i's logits: softmax and loss are unchanged, and since each row
    # of dz sums to zero, dh = dz (W + 1 c^T) is unchanged too.
    loss2, dh2, _ = alst.ce_fwd_bwd(h, W, labels, 1.0)
    c = np.random.default_rng(11).standard_normal(W.shape[1])
    loss3, dh3, _ = alst.ce_fwd_bwd(h, W + c[None, :], labels, 1.0)
    np.testing.assert_allclose(loss3, loss2, atol=1e-12)
    np.testing.assert_allclose(dh3, dh2, atol=1e-12)


@pytest.mark.parametrize("bf16", [False, True])
def test_tiled_equals_untiled(bf16):
    x, Wgu, Wd, dy = _mlp_inputs(seed=4, L=37)
    y0, h0 = alst.mlp_fwd(x, Wgu, Wd, bf16)
    dx0, a0, b0 = alst.mlp_bwd(x, Wgu, Wd, dy, bf16)
    for T in (8, 16, 37):
        y, dx, a, b = alst.mlp_tiled(x, Wgu, Wd, dy, T, bf16)
        # row-wise outputs: same arithmetic up to the BLAS kernel's blocking
        np.testing.assert_allclose(y, y0, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(dx, dx0, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(a, a0, atol=1e-12)  # sums over tokens, re-associated
        np.testing.assert_allclose(b, b0, atol=1e-12)
    h, W, labels = _ce_inputs(seed=5)
    l0, g0, w0 = alst.ce_fwd_bwd(h, W, labels, 0.25, bf16)
    for T in (5, 16, 33):
        l, g, w = alst.ce_tiled(h, W, labels, 0.25, T, bf16)
        np.testing.assert_allclose(l, l0, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(g, g0, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(w, w0, atol=1e-13)


def test_bf16_operand_mlp_rounds_exactly_the_stated_intermediates():
    """With bf16_operands, H, dH and [dG | dU] (and nothing else) go through
    torch's bf16 conversion; the result differs from the exact MLP at the
    bf16 level."""
    x, Wgu, Wd, dy = _mlp_inputs(seed=6)
    F = Wd.shape[1]
    bf = lambda a: torch.tensor(a).to(torch.bfloat16).double().numpy()
    gu = x @ Wgu.T
    g, u = gu[:, :F], gu[:, F:]
    s = 1 / (1 + np.exp(-g))
    h = bf(g * s * u)
    dh = bf(dy @ Wd)
    dgu = bf(np.concatenate([dh * u * s * (1 + g * (1 - s)), dh * g * s], 1))
    y, hb = alst.mlp_fwd(x, Wgu, Wd, bf16_operands=True)
    np.testing.assert_array_equal(hb, h)
    np.testing.assert_allclose(y, h @ Wd.T, atol=1e-13)
    dx, dWgu, dWd = alst.mlp_bwd(x, Wgu, Wd, dy, bf16_operands=True)
    np.testing.assert_allclose(dx, dgu @ Wgu, atol=1e-12)
    np.testing.assert_allclose(dWgu, dgu.T @ x, atol=1e-12)
    np.testing.assert_allclose(dWd, dy.T @ h, atol=1e-12)
    ye, _ = alst.mlp_fwd(x, Wgu, Wd)
    assert 1e-6 < np.linalg.norm(y - ye) / np.linalg.norm(ye) < 1e-2
    assert np.array_equal(bf16_round(h), h)


def test_row_checks_without_weight_gradients_agree():
    x, Wgu, Wd, dy = _mlp_inputs(seed=7)
    a = alst.mlp_bwd(x, Wgu, Wd, dy, True)
    b = alst.mlp_bwd(x, Wgu, Wd, dy, True, weight_grads=False)
    np.testing.assert_array_equal(a[0], b[0])
    assert b[1] is None and b[2] is None
    h, W, labels = _ce_inputs(seed=8)
    a = alst.ce_fwd_bwd(h, W, labels, 0.5, True)
    b = alst.ce_fwd_bwd(h, W, labels, 0.5, True, weight_grad=False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert b[2] is None


def test_tile_bytes_scale_with_the_tile():
    a, b = alst.tile_bytes(4096, 4096, 14336, 128256), alst.tile_bytes(65536, 4096, 14336, 128256)
    assert b["mlp_bwd"] == 16 * a["mlp_bwd"] and b["ce"] == 16 * a["ce"]
