"""The parity tolerance accepts what a bf16-operand backward can reach and
rejects a wrong one (CPU only).

The emulation computes the layer backward in fp64 with exactly the roundings
a tensor-core implementation makes: Q, K, V, O, dO and the softmax tiles P and
dS rounded to bf16 before every product that consumes them.  Its error against
the exact oracle must pass tests/tolerance.py; the same emulation with the
Delta term dropped from dS must fail it.
"""

import math

import numpy as np
import torch

from headwise_chunked_context_gb300 import synth
from oracle import upipe_oracle as orc
from tests.tolerance import assert_close


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).double().numpy()


def _emulated_bwd(x, w, wo, dout, H, Hkv, theta, drop_delta=False):
    L = x.shape[0]
    d = wo.shape[1] // H
    g = H // Hkv
    pos = np.arange(L)
    q, k, v = (_bf(t) for t in orc.project_qkv(x, w, H, Hkv, d, theta))
    o, lse = orc.attention_core_fwd(q, k, v)
    o = _bf(o)
    do = _bf((dout @ wo).reshape(L, H, d))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    scale = 1 / math.sqrt(d)
    for h in range(H):
        kh, vh = k[:, h // g], v[:, h // g]
        delta = 0.0 if drop_delta else np.sum(do[:, h] * o[:, h], 1)[:, None]
        P = np.exp(q[:, h] @ kh.T * scale - lse[h][:, None])
        P[np.triu_indices(L, 1)] = 0
        dS = _bf(P * (do[:, h] @ vh.T - delta))
        dv[:, h // g] += _bf(P).T @ do[:, h]
        dk[:, h // g] += dS.T @ q[:, h] * scale
        dq[:, h] = dS @ kh * scale
    dq = orc.rope_apply(dq, pos, theta, inverse=True)
    dk = orc.rope_apply(dk, pos, theta, inverse=True)
    dqkv = np.concatenate([dq.reshape(L, -1), dk.reshape(L, -1), dv.reshape(L, -1)], 1)
    return dqkv @ w, dqkv.T @ x


def test_tolerance_accepts_bf16_operand_backward_and_rejects_a_dropped_term():
    s = synth.LayerShape(L=512, D=512, H=8, Hkv=2)
    x, w, wo, dout = (t.double().numpy() for t in synth.layer_inputs(s))
    dx, dw, _ = orc.layer_bwd(x, w, wo, dout, s.H, s.Hkv, s.theta)
    edx, edw = _emulated_bwd(x, w, wo, dout, s.H, s.Hkv, s.theta)
    assert_close(edx, dx, "dx")
    assert_close(edw, dw, "dWqkv", weight_grad=True)
    bdx, bdw = _emulated_bwd(x, w, wo, dout, s.H, s.Hkv, s.theta, drop_delta=True)
    failed = 0
    for got, ref, n, wg in ((bdx, dx, "dx", False), (bdw, dw, "dWqkv", True)):
        try:
            assert_close(got, ref, n, weight_grad=wg)
        except AssertionError:
            failed += 1
    assert failed == 2
