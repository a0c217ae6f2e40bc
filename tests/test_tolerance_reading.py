"""The parity tolerance accepts what an fp32-accumulate implementation of
the precision model reaches and rejects a wrong one (CPU only).

"bf16 in / fp32 accumulate": an implementation rounds every contraction
input to bf16 and accumulates in fp32.  The emulation below does exactly
that in NumPy float32 (bf16 rounding of Q, K, V, O, dO, P and dS through
torch's conversion; float32 products and sums), independently of the
oracle's code.  Against the oracle's fp64 precision-model mode it must pass
tests/tolerance.py (weight gradients scaled by max(1, RMS)); against the
plain fp64 definition it must pass the triangle bound; with the Delta term
dropped from dS (a mistake planted here, on the CPU) it must fail.
"""

import math

import numpy as np
import torch

from headwise_chunked_context_gb300 import synth
from oracle import upipe_oracle as orc
from tests.tolerance import assert_close, assert_close_plain

F32 = np.float32


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _emulated_layer(x, w, wo, dout, H, Hkv, theta, drop_delta=False):
    """float32 layer forward + backward with bf16 contraction inputs."""
    L = x.shape[0]
    d = wo.shape[1] // H
    g = H // Hkv
    pos = np.arange(L)
    x32, w32, wo32, dout32 = (a.astype(F32) for a in (x, w, wo, dout))
    qkv = x32 @ w32.T
    q, k, v = orc.split_qkv(qkv, H, Hkv, d)
    q = _bf(orc.rope_apply(q.astype(np.float64), pos, theta))
    k = _bf(orc.rope_apply(k.astype(np.float64), pos, theta))
    v = _bf(v)
    scale = F32(1 / math.sqrt(d))
    causal = np.tril(np.ones((L, L), dtype=bool))
    o = np.zeros((L, H, d), F32)
    lse = np.zeros((H, L), F32)
    for h in range(H):
        S = (q[:, h] @ k[:, h // g].T) * scale
        S = np.where(causal, S, -np.inf).astype(F32)
        m = S.max(1)
        lse[h] = m + np.log(np.exp(S - m[:, None]).sum(1))
        o[:, h] = _bf(np.exp(S - lse[h][:, None])) @ v[:, h // g]
    o = _bf(o)
    out = o.reshape(L, -1) @ wo32.T
    do = _bf((dout32 @ wo32).reshape(L, H, d))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(H):
        kh, vh = k[:, h // g], v[:, h // g]
        delta = F32(0) if drop_delta else np.sum(do[:, h] * o[:, h], 1)[:, None]
        P = np.where(causal, np.exp((q[:, h] @ kh.T) * scale - lse[h][:, None]), F32(0)).astype(F32)
        dS = _bf(P * (do[:, h] @ vh.T - delta))
        dv[:, h // g] += _bf(P).T @ do[:, h]
        dk[:, h // g] += (dS.T @ q[:, h]) * scale
        dq[:, h] = (dS @ kh) * scale
    dq = orc.rope_apply(dq.astype(np.float64), pos, theta, inverse=True).astype(F32)
    dk = orc.rope_apply(dk.astype(np.float64), pos, theta, inverse=True).astype(F32)
    dqkv = np.concatenate([dq.reshape(L, -1), dk.reshape(L, -1), dv.reshape(L, -1)], 1)
    return out, lse, dqkv @ w32, dqkv.T @ x32, dout32.T @ o.reshape(L, -1)


def test_tolerance_accepts_fp32_accumulate_and_rejects_a_dropped_term():
    s = synth.LayerShape(L=512, D=512, H=8, Hkv=2)
    x, w, wo, dout = (t.double().numpy() for t in synth.layer_inputs(s))
    args = (x, w, wo, s.H, s.Hkv, s.theta)
    m_out, m_lse, _ = orc.layer_fwd(*args, bf16_operands=True)
    model = (m_out, m_lse, *orc.layer_bwd(x, w, wo, dout, s.H, s.Hkv, s.theta, bf16_operands=True))
    p_out, p_lse, _ = orc.layer_fwd(*args)
    plain = (p_out, p_lse, *orc.layer_bwd(x, w, wo, dout, s.H, s.Hkv, s.theta))
    names = ("out", "lse", "dx", "dWqkv", "dWo")
    wgrad = (False, False, False, True, True)
    emu = _emulated_layer(x, w, wo, dout, s.H, s.Hkv, s.theta)
    for got, m, p, n, wg in zip(emu, model, plain, names, wgrad):
        assert_close(got, m, n, weight_grad=wg)
        assert_close_plain(got, p, m, n, weight_grad=wg)
    bad = _emulated_layer(x, w, wo, dout, s.H, s.Hkv, s.theta, drop_delta=True)
    failed = []
    for got, m, n, wg in list(zip(bad, model, names, wgrad))[2:]:
        try:
            assert_close(got, m, n, weight_grad=wg)
        except AssertionError:
            failed.append(n)
    assert failed == ["dx", "dWqkv"], failed
