"""fp64 CPU oracle for the sequence-tiled MLP and loss around the attention
layer (ALST-style tiling).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: it is used by ``tests/`` only.  It shares no code with
the CUDA path; both sides only share the seeded input generator
(``synth``), which holds no arithmetic.

What it computes, and where that is stated
------------------------------------------
"Untied Ulysses Pushes Llama-3-8B Training to 5 Million Tokens" (orply.com
talk write-up), paragraph on Arctic Long Sequence Training: element-wise and
sequence-wide computations -- the MLPs and the loss -- need no buffer that
spans the whole sequence at once; they are computed tile by tile along the
sequence axis.  Tiling changes where the intermediates live, not what is
computed, so the oracle is the plain definition of each operator, plus a
tiled restatement pinned to it.

Readings of points the pages leave open:

* MLP: the models the pages train (Llama-3-8B, the 32B Qwen family) use the
  gated SiLU ("SwiGLU") MLP without biases:
  ``y = (silu(x Wg^T) * (x Wu^T)) Wd^T``, silu(g) = g * sigmoid(g).  The
  gate and up weights are one matrix ``Wgu = [Wg; Wu]`` ([2F, D]: the F
  gate rows, then the F up rows).
* Loss: per-token cross-entropy of the LM head, ``z = h W^T`` over the
  vocabulary, ``loss_i = logsumexp(z_i) - z_i[label_i]``; labels are given
  (the caller shifts them), a negative label marks a token that contributes
  nothing; the backward is the gradient of ``sum_i scale * loss_i`` for a
  caller-given ``scale`` (1 / valid tokens gives the mean).
* Precision model (``bf16_operands=True``, as in the attention oracle):
  every input of every contraction is rounded to bf16 -- the stored
  intermediates H = silu(g) * u, dH = dy Wd, dG / dU and dZ -- and every
  product, sum and element-wise step stays exact fp64.
"""

from __future__ import annotations

import numpy as np

from oracle.upipe_oracle import bf16_round

F64 = np.float64


def _op(a, bf16_operands):
    return bf16_round(a) if bf16_operands else a


def _sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


# ---------------------------------------------------------------------------
# SwiGLU MLP
# ---------------------------------------------------------------------------

def mlp_fwd(x, Wgu, Wd, bf16_operands=False):
    """y [L, D] and the hidden activation H [L, F] of the SwiGLU MLP."""
    x = np.asarray(x, dtype=F64)
    Wgu = np.asarray(Wgu, dtype=F64)
    Wd = np.asarray(Wd, dtype=F64)
    F = Wd.shape[1]
    gu = x @ Wgu.T
    g, u = gu[:, :F], gu[:, F:]
    h = _op(g * _sigmoid(g) * u, bf16_operands)
    return h @ Wd.T, h


def mlp_bwd(x, Wgu, Wd, dy, bf16_operands=False, weight_grads=True):
    """dx [L, D], dWgu [2F, D], dWd [D, F]: gradient of sum(y * dy).

    silu'(g) = s (1 + g (1 - s)), s = sigmoid(g).  Under the precision
    model H, dH = dy Wd and [dG | dU] enter their products as bf16.  With
    weight_grads=False only dx is formed (the other two are None), for
    checks of sampled rows.
    """
    x = np.asarray(x, dtype=F64)
    Wgu = np.asarray(Wgu, dtype=F64)
    Wd = np.asarray(Wd, dtype=F64)
    dy = np.asarray(dy, dtype=F64)
    F = Wd.shape[1]
    gu = x @ Wgu.T
    g, u = gu[:, :F], gu[:, F:]
    s = _sigmoid(g)
    silu = g * s
    h = _op(silu * u, bf16_operands)
    dh = _op(dy @ Wd, bf16_operands)
    dg = dh * u * (s * (1.0 + g * (1.0 - s)))
    du = dh * silu
    dgu = _op(np.concatenate([dg, du], axis=1), bf16_operands)
    if not weight_grads:
        return dgu @ Wgu, None, None
    return dgu @ Wgu, dgu.T @ x, dy.T @ h


def mlp_tiled(x, Wgu, Wd, dy, T, bf16_operands=False):
    """The same operator computed T rows at a time: each tile's outputs come
    from that tile's rows alone, and the weight gradients are the sum of the
    tiles' contributions.  Returns (y, dx, dWgu, dWd)."""
    L = x.shape[0]
    ys, dxs = [], []
    dWgu = dWd = 0.0
    for r0 in range(0, L, T):
        sl = slice(r0, min(L, r0 + T))
        y, _ = mlp_fwd(x[sl], Wgu, Wd, bf16_operands)
        dx, a, b = mlp_bwd(x[sl], Wgu, Wd, dy[sl], bf16_operands)
        ys.append(y)
        dxs.append(dx)
        dWgu = dWgu + a
        dWd = dWd + b
    return np.concatenate(ys), np.concatenate(dxs), dWgu, dWd


# ---------------------------------------------------------------------------
# Cross-entropy loss of the LM head
# ---------------------------------------------------------------------------

def ce_fwd_bwd(h, W, labels, scale, bf16_operands=False, weight_grad=True):
    """Per-token loss [L] (0 where label < 0), dh [L, D] and dW [V, D] (None
    with weight_grad=False, for checks of sampled rows), the gradients of
    sum_i scale * loss_i.

    z = h W^T; loss_i = logsumexp(z_i) - z_i[label_i];
    dz_ij = scale * (softmax(z_i)_j - [j == label_i]) for a valid token, 0
    otherwise.  Under the precision model dz enters its products as bf16.
    """
    h = np.asarray(h, dtype=F64)
    W = np.asarray(W, dtype=F64)
    labels = np.asarray(labels)
    z = h @ W.T
    zmax = z.max(axis=1, keepdims=True)
    lse = (zmax + np.log(np.exp(z - zmax).sum(axis=1, keepdims=True)))[:, 0]
    valid = labels >= 0
    rows = np.arange(z.shape[0])
    lab = np.where(valid, labels, 0)
    loss = np.where(valid, lse - z[rows, lab], 0.0)
    p = np.exp(z - lse[:, None])
    p[rows[valid], lab[valid]] -= 1.0
    dz = _op(np.where(valid[:, None], scale * p, 0.0), bf16_operands)
    return loss, dz @ W, (dz.T @ h if weight_grad else None)


def ce_tiled(h, W, labels, scale, T, bf16_operands=False):
    """ce_fwd_bwd computed T rows at a time (dW summed over the tiles)."""
    L = h.shape[0]
    losses, dhs = [], []
    dW = 0.0
    for r0 in range(0, L, T):
        sl = slice(r0, min(L, r0 + T))
        loss, dh, dw = ce_fwd_bwd(h[sl], W, labels[sl], scale, bf16_operands)
        losses.append(loss)
        dhs.append(dh)
        dW = dW + dw
    return np.concatenate(losses), np.concatenate(dhs), dW


def tile_bytes(T: int, D: int, F: int, V: int, elem: int = 2) -> dict:
    """Intermediate bytes one tile of T rows holds, by operator: the MLP's
    backward keeps H, dH ([T, F]) and dG|dU ([T, 2F]); the loss keeps the
    logits [T, V] in fp32 and dZ [T, V].  Untiled, T = L."""
    return {"mlp_bwd": T * F * elem * 4, "ce": T * V * (4 + elem)}
