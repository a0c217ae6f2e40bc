"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test fixes the oracle to something independent of its own code:
hand-worked closed forms (tests/golden/closed_forms.txt), a library
attention (torch's scaled_dot_product_attention in float64), scipy's
logsumexp, central finite differences of the forward, torch autograd of a
float64 layer written with complex-number RoPE, and invariants that the
definition implies (softmax rows sum to 1, RoPE preserves norms and depends
only on relative position, GQA equals explicit KV repetition, every chunk
size U gives the same layer).  A dropped term, a wrong sign or index, or a
transposed operand in the oracle breaks at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import upipe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def _eval(expr):
    env = {"exp": math.exp, "log": math.log, "cos": math.cos, "sin": math.sin, "sqrt": math.sqrt}
    return float(eval(expr, {"__builtins__": {}}, env))


def _mat(s):
    return np.array([[_eval(e) for e in row.split(",")] for row in s.split(";")], dtype=np.float64)


def _golden_cases():
    cases, cur = {}, None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = [t.strip() for t in line.split(":", 1)]
        if key == "case":
            cur = cases.setdefault(val, {})
        else:
            cur[key] = val
    return cases


GOLD = _golden_cases()


# --------------------------------------------------------------------- golden

@pytest.mark.parametrize("name", ["two_token_attention", "uniform_scores"])
def test_attention_closed_forms(name):
    c = GOLD[name]
    q, k, v = _mat(c["q"]), _mat(c["k"]), _mat(c["v"])
    o, lse = orc.attention_core_fwd(q[:, None], k[:, None], v[:, None])
    np.testing.assert_allclose(o[:, 0], _mat(c["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], _mat(c["lse"])[0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("name", ["rope_d2", "rope_d4"])
def test_rope_closed_forms(name):
    c = GOLD[name]
    x = _mat(c["x"])
    pos = [int(p) for p in c["positions"].split(",")]
    out = orc.rope_apply(x[:, None, :], pos, float(c["theta"]))[:, 0]
    np.testing.assert_allclose(out, _mat(c["out"]), rtol=0, atol=1e-13)


# ------------------------------------------------------------ library pins

def _sdpa_gqa(q, k, v):
    """torch SDPA (float64, causal) with KV heads repeated for GQA."""
    H, Hkv = q.shape[1], k.shape[1]
    g = H // Hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(np.repeat(k, g, axis=1)).permute(1, 0, 2)[None]
    tv = torch.from_numpy(np.repeat(v, g, axis=1)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("L,H,Hkv,d", [(37, 4, 2, 16), (64, 8, 1, 32), (5, 2, 2, 8)])
def test_core_fwd_matches_library_attention(L, H, Hkv, d):
    rng = np.random.default_rng(11)
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    o, lse = orc.attention_core_fwd(q, k, v)
    np.testing.assert_allclose(o, _sdpa_gqa(q, k, v), rtol=1e-11, atol=1e-12)
    g = H // Hkv
    for h in range(H):
        S = q[:, h] @ k[:, h // g].T / math.sqrt(d)
        S[np.triu_indices(L, 1)] = -np.inf
        np.testing.assert_allclose(lse[h], logsumexp(S, axis=1), rtol=1e-13, atol=1e-12)


def test_row0_and_zero_query_closed_forms():
    rng = np.random.default_rng(3)
    L, d = 50, 16
    q = rng.standard_normal((L, 1, d))
    k = rng.standard_normal((L, 1, d))
    v = rng.standard_normal((L, 1, d))
    o, lse = orc.attention_core_fwd(q, k, v)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], q[0, 0] @ k[0, 0] / math.sqrt(d), atol=1e-13)
    o0, lse0 = orc.attention_core_fwd(np.zeros_like(q), k, v)
    prefix_mean = np.cumsum(v[:, 0], axis=0) / np.arange(1, L + 1)[:, None]
    np.testing.assert_allclose(o0[:, 0], prefix_mean, atol=1e-13)
    np.testing.assert_allclose(lse0[0], np.log(np.arange(1, L + 1)), atol=1e-13)


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(5)
    L, d = 40, 8
    q = rng.standard_normal((L, 2, d)) * 3
    k = rng.standard_normal((L, 1, d)) * 3
    v = rng.standard_normal((L, 1, d))
    _, lse = orc.attention_core_fwd(q, k, v)
    for h in range(2):
        S = q[:, h] @ k[:, 0].T / math.sqrt(d)
        P = np.exp(S - lse[h][:, None])
        P[np.triu_indices(L, 1)] = 0.0
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)


# ------------------------------------------------------------------- RoPE

def test_rope_invariants():
    rng = np.random.default_rng(7)
    L, nh, d, theta = 33, 3, 16, 500000.0
    x = rng.standard_normal((L, nh, d))
    pos = np.arange(L)
    y = orc.rope_apply(x, pos, theta)
    # pairwise norms preserved
    nx = x[..., : d // 2] ** 2 + x[..., d // 2:] ** 2
    ny = y[..., : d // 2] ** 2 + y[..., d // 2:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12)
    # position 0 and theta -> inf (all but pair 0 frozen) are the identity
    np.testing.assert_allclose(y[0], x[0], atol=0)
    # inverse undoes forward
    np.testing.assert_allclose(orc.rope_apply(y, pos, theta, inverse=True), x, atol=1e-12)
    # q_m . k_n depends only on m - n
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    for m, n, s in [(5, 2, 100), (17, 17, 1000), (3, 9, 12345)]:
        a = orc.rope_apply(q, [m], theta)[0, 0] @ orc.rope_apply(k, [n], theta)[0, 0]
        b = orc.rope_apply(q, [m + s], theta)[0, 0] @ orc.rope_apply(k, [n + s], theta)[0, 0]
        assert abs(a - b) < 1e-10


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(8)
    L, d, theta = 20, 8, 500000.0
    x = rng.standard_normal((L, 1, d))
    pos = np.arange(L) * 1000 + 7
    z = x[:, 0, : d // 2] + 1j * x[:, 0, d // 2:]
    freqs = theta ** (-np.arange(0, d, 2) / d)
    zr = z * np.exp(1j * pos[:, None] * freqs[None, :])
    y = orc.rope_apply(x, pos, theta)[:, 0]
    np.testing.assert_allclose(y[:, : d // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(y[:, d // 2:], zr.imag, atol=1e-12)


# --------------------------------------------------------------- projections

def test_qkv_row_order_one_hot():
    """A single 1 at row (v head 1, dim 3), column j copies x[:, j] there."""
    L, D, H, Hkv, d = 6, 5, 4, 2, 4
    x = np.random.default_rng(1).standard_normal((L, D))
    W = np.zeros(((H + 2 * Hkv) * d, D))
    W[(H + Hkv + 1) * d + 3, 2] = 1.0
    W[(1) * d + 0, 4] = 1.0  # q head 1, dim 0 (rotated with dim 2 by RoPE)
    q, k, v = orc.project_qkv(x, W, H, Hkv, d, 500000.0, rope=False)
    np.testing.assert_array_equal(v[:, 1, 3], x[:, 2])
    assert np.count_nonzero(v) == np.count_nonzero(x[:, 2])
    np.testing.assert_array_equal(q[:, 1, 0], x[:, 4])
    assert np.count_nonzero(k) == 0


# ---------------------------------------------------------------- GQA

def test_gqa_equals_repeated_kv_layer():
    rng = np.random.default_rng(9)
    L, D, H, Hkv, d = 24, 16, 4, 2, 8
    x = rng.standard_normal((L, D))
    Wqkv = rng.standard_normal(((H + 2 * Hkv) * d, D)) * 0.3
    Wo = rng.standard_normal((D, H * d)) * 0.3
    g = H // Hkv
    Wq = Wqkv[: H * d]
    Wk = Wqkv[H * d:(H + Hkv) * d].reshape(Hkv, d, D)
    Wv = Wqkv[(H + Hkv) * d:].reshape(Hkv, d, D)
    W_mha = np.concatenate([Wq, np.repeat(Wk, g, axis=0).reshape(-1, D), np.repeat(Wv, g, axis=0).reshape(-1, D)])
    out_g, lse_g, _ = orc.layer_fwd(x, Wqkv, Wo, H, Hkv, 1e4)
    out_m, lse_m, _ = orc.layer_fwd(x, W_mha, Wo, H, H, 1e4)
    np.testing.assert_allclose(out_g, out_m, atol=1e-12)
    np.testing.assert_allclose(lse_g, lse_m, atol=1e-12)


# ---------------------------------------------------------------- backward

def _micro(seed=0, L=16, D=32, H=4, Hkv=2, d=8):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((L, D))
    Wqkv = rng.standard_normal(((H + 2 * Hkv) * d, D)) * 0.2
    Wo = rng.standard_normal((D, H * d)) * 0.2
    dout = rng.standard_normal((L, D))
    return x, Wqkv, Wo, dout, H, Hkv, 50.0


def test_backward_matches_finite_differences():
    x, Wqkv, Wo, dout, H, Hkv, theta = _micro()
    dx, dWqkv, dWo = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta)

    def f(x_, Wqkv_, Wo_):
        return float(np.sum(orc.layer_fwd(x_, Wqkv_, Wo_, H, Hkv, theta)[0] * dout))

    rng = np.random.default_rng(1)
    h = 1e-6
    for name, arr, grad in [("x", x, dx), ("Wqkv", Wqkv, dWqkv), ("Wo", Wo, dWo)]:
        idx = [tuple(rng.integers(0, s) for s in arr.shape) for _ in range(12)]
        for ix in idx:
            plus, minus = arr.copy(), arr.copy()
            plus[ix] += h
            minus[ix] -= h
            args_p = [plus if n == name else a for n, a in (("x", x), ("Wqkv", Wqkv), ("Wo", Wo))]
            args_m = [minus if n == name else a for n, a in (("x", x), ("Wqkv", Wqkv), ("Wo", Wo))]
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            assert abs(fd - grad[ix]) <= 1e-6 * max(1.0, abs(fd)), (name, ix, fd, grad[ix])


def _torch_layer(x, Wqkv, Wo, H, Hkv, theta):
    """float64 torch layer: complex-number RoPE and library SDPA."""
    L, D = x.shape
    d = Wo.shape[1] // H
    g = H // Hkv
    qkv = x @ Wqkv.T
    q = qkv[:, : H * d].reshape(L, H, d)
    k = qkv[:, H * d:(H + Hkv) * d].reshape(L, Hkv, d)
    v = qkv[:, (H + Hkv) * d:].reshape(L, Hkv, d)
    freqs = theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(L, d // 2, dtype=torch.float64),
                      torch.arange(L, dtype=torch.float64)[:, None] * freqs[None])

    def rope(t):
        z = torch.complex(t[..., : d // 2], t[..., d // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    q, k = rope(q), rope(k)
    k = k.repeat_interleave(g, dim=1)
    v = v.repeat_interleave(g, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None], v.permute(1, 0, 2)[None], is_causal=True)
    return o[0].permute(1, 0, 2).reshape(L, H * d) @ Wo.T


@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (2, 2)])
def test_layer_matches_torch_autograd(H, Hkv):
    x, Wqkv, Wo, dout, _, _, theta = _micro(seed=4, H=H, Hkv=Hkv)
    out, _, _ = orc.layer_fwd(x, Wqkv, Wo, H, Hkv, theta)
    dx, dWqkv, dWo = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta)
    tx, tW, tWo = (torch.tensor(a, requires_grad=True) for a in (x, Wqkv, Wo))
    tout = _torch_layer(tx, tW, tWo, H, Hkv, theta)
    (tout * torch.from_numpy(dout)).sum().backward()
    np.testing.assert_allclose(out, tout.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dWqkv, tW.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dWo, tWo.grad.numpy(), rtol=1e-9, atol=1e-11)


# ------------------------------------------------------------- chunking

@pytest.mark.parametrize("H,Hkv,Us", [(4, 2, (1, 2, 4)), (8, 2, (1, 2, 4, 8)), (4, 4, (1, 2, 4))])
def test_every_chunk_size_gives_the_plain_layer(H, Hkv, Us):
    x, Wqkv, Wo, dout, _, _, theta = _micro(seed=2, H=H, Hkv=Hkv, L=20, D=24)
    out, lse, _ = orc.layer_fwd(x, Wqkv, Wo, H, Hkv, theta)
    dx, dWqkv, dWo = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta)
    for U in Us:
        out_c, lse_c = orc.layer_fwd_chunked(x, Wqkv, Wo, H, Hkv, theta, U)
        dx_c, dWqkv_c, dWo_c = orc.layer_bwd_chunked(x, Wqkv, Wo, dout, H, Hkv, theta, U)
        for a, b in [(out, out_c), (lse, lse_c), (dx, dx_c), (dWqkv, dWqkv_c), (dWo, dWo_c)]:
            np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------ sampled-row helpers

def test_sampled_rows_agree_with_full():
    rng = np.random.default_rng(6)
    L, H, Hkv, d = 300, 4, 1, 16
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    do = rng.standard_normal((L, H, d))
    o, lse = orc.attention_core_fwd(q, k, v)
    dq, dk, dv = orc.attention_core_bwd(q, k, v, o, lse, do)
    scale = 1.0 / math.sqrt(d)
    rows = np.array([0, 1, 128, 255, 299])
    h = 2
    orow, lrow = orc.attention_head_rows(q[rows, h], rows, k[:, 0], v[:, 0], scale)
    np.testing.assert_allclose(orow, o[rows, h], atol=1e-13)
    np.testing.assert_allclose(lrow, lse[h, rows], atol=1e-13)
    dqr = orc.attention_dq_rows(q[rows, h], rows, k[:, 0], v[:, 0], do[rows, h], o[rows, h], lse[h, rows], scale)
    np.testing.assert_allclose(dqr, dq[rows, h], atol=1e-12)
    T = 40
    dk_t = np.zeros((T, d))
    dv_t = np.zeros((T, d))
    for hh in range(H):
        a, b = orc.attention_dkv_tail(q[-T:, hh], k[-T:, 0], v[-T:, 0], do[-T:, hh], o[-T:, hh], lse[hh, -T:], scale)
        dk_t += a
        dv_t += b
    np.testing.assert_allclose(dk_t, dk[-T:, 0], atol=1e-12)
    np.testing.assert_allclose(dv_t, dv[-T:, 0], atol=1e-12)


# ------------------------------------------------------- memory arithmetic

def test_intermediate_memory_ratio():
    # U >= g: chunk buffers are exactly U/H of the unchunked ones.
    for (H, Hkv, U) in [(32, 8, 8), (64, 8, 16), (64, 8, 8), (32, 8, 4)]:
        L, d = 131072, 128
        r = orc.intermediate_bytes(L, U, H, Hkv, d) / orc.intermediate_bytes(L, H, H, Hkv, d)
        assert r == pytest.approx(U / H, abs=0)
    # 32B-shaped layer (H=64, Hkv=8), U=8: 87.5% less intermediate memory,
    # the figure the abstract quotes for 32B Transformers.
    r = orc.intermediate_bytes(131072, 8, 64, 8, 128) / orc.intermediate_bytes(131072, 64, 64, 8, 128)
    assert 1 - r == pytest.approx(0.875, abs=0)
    # U < g: each chunk still needs its one KV head.
    assert orc.intermediate_bytes(1024, 2, 8, 2, 128) == 1024 * 128 * 2 * (4 + 2)


# ----------------------------------------------------- bf16 precision model

def test_bf16_round_matches_library_conversion():
    rng = np.random.default_rng(12)
    a = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40]])
    # exact ties: 1 + 2^-8 (tie, even stays at 1) and 1 + 3*2^-8 (tie, rounds up)
    a = np.concatenate([a, [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)]])
    want = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(orc.bf16_round(a), want)
    assert orc.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert orc.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6


def _bf(a):
    """bf16 rounding through torch's own conversion (independent of
    orc.bf16_round)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).float().to(torch.bfloat16).double().numpy()


def test_bf16_operand_layer_is_the_exact_layer_with_rounded_contraction_inputs():
    """With bf16_operands the layer equals a restatement written here from
    the definition, whose every contraction input (Q, K, V after RoPE, O,
    dO; P in the backward's recomputation of O from the LSE and in P^T dO;
    dS in dS K and dS^T Q) goes through torch's bf16 conversion, with all
    else exact (the forward output's own P V keeps P exact); and it differs
    from the exact layer only at the bf16 level."""
    x, Wqkv, Wo, dout, H, Hkv, theta = _micro(seed=3, L=24, D=32)
    L = x.shape[0]
    d = Wo.shape[1] // H
    g = H // Hkv
    sc = 1 / math.sqrt(d)
    out_b, lse_b, o_b = orc.layer_fwd(x, Wqkv, Wo, H, Hkv, theta, bf16_operands=True)
    dx_b, dW_b, dWo_b = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta, bf16_operands=True)
    q, k, v = (_bf(t) for t in orc.project_qkv(x, Wqkv, H, Hkv, d, theta))
    o = np.zeros((L, H, d))
    lse = np.zeros((H, L))
    causal = np.tril(np.ones((L, L), dtype=bool))
    o_fwd = np.zeros((L, H, d))
    for h in range(H):
        S = q[:, h] @ k[:, h // g].T * sc
        S[~causal] = -np.inf
        lse[h] = logsumexp(S, axis=1)
        P = np.exp(S - lse[h][:, None])
        o_fwd[:, h] = P @ v[:, h // g]
        o[:, h] = _bf(P) @ v[:, h // g]
    o_fwd = _bf(o_fwd)
    o = _bf(o)
    do = _bf((dout @ Wo).reshape(L, H, d))
    pos = np.arange(L)

    def grads(o_used):
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for h in range(H):
            S = q[:, h] @ k[:, h // g].T * sc
            P = np.where(causal, np.exp(S - lse[h][:, None]), 0.0)
            delta = np.sum(do[:, h] * o_used[:, h], axis=1)
            dS = _bf(P * (do[:, h] @ v[:, h // g].T - delta[:, None]))
            dv[:, h // g] += _bf(P).T @ do[:, h]
            dk[:, h // g] += dS.T @ q[:, h] * sc
            dq[:, h] = dS @ k[:, h // g] * sc
        dqkv = np.concatenate([orc.rope_apply(dq, pos, theta, inverse=True).reshape(L, -1),
                               orc.rope_apply(dk, pos, theta, inverse=True).reshape(L, -1), dv.reshape(L, -1)], 1)
        return dqkv @ Wqkv, dqkv.T @ x, dout.T @ o_used.reshape(L, -1)

    np.testing.assert_allclose(lse_b, lse, atol=1e-13)
    np.testing.assert_allclose(o_b, o_fwd, atol=1e-13)
    np.testing.assert_allclose(out_b, o_fwd.reshape(L, -1) @ Wo.T, atol=1e-13)
    for got, ref in zip((dx_b, dW_b, dWo_b), grads(o)):
        np.testing.assert_allclose(got, ref, atol=1e-12)
    # O kept from the forward: the backward reads the forward's own output
    kept = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta, bf16_operands=True, kept_o=True)
    for got, ref in zip(kept, grads(o_fwd)):
        np.testing.assert_allclose(got, ref, atol=1e-12)
    assert np.abs(kept[2] - dWo_b).max() > 0  # the two O differ at the bf16 level
    for a_, b_ in zip(orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta, kept_o=True),
                      orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta)):
        np.testing.assert_array_equal(a_, b_)  # without the model both are the exact O
    out, _, _ = orc.layer_fwd(x, Wqkv, Wo, H, Hkv, theta)
    rel = np.linalg.norm(out_b - out) / np.linalg.norm(out)
    assert 1e-5 < rel < 1e-2
    dx, dW, dWo = orc.layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta)
    for a_, b_ in ((dx_b, dx), (dW_b, dW), (dWo_b, dWo)):
        assert 1e-6 < np.linalg.norm(a_ - b_) / np.linalg.norm(b_) < 1e-2


# ------------------------------------------------- streamed query-row blocks
#
# The attention functions stream query rows in blocks (sized so one block's
# scores stay near 64 MB).  At the sizes above every call is one block; the
# tests below force several blocks, with a ragged last one, so that the
# multi-block path (each block's mask offset and key range) is pinned too.

@pytest.fixture
def small_blocks(monkeypatch):
    monkeypatch.setattr(orc, "ROW_BLOCK", 37)
    assert orc._row_block(300, 300) == 37


@pytest.mark.parametrize("L,H,Hkv,d", [(300, 4, 2, 16), (111, 2, 1, 8)])
def test_multi_block_core_forward_matches_library_attention(small_blocks, L, H, Hkv, d):
    rng = np.random.default_rng(21)
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    o, lse = orc.attention_core_fwd(q, k, v)
    np.testing.assert_allclose(o, _sdpa_gqa(q, k, v), rtol=1e-11, atol=1e-12)
    g = H // Hkv
    for h in range(H):
        S = q[:, h] @ k[:, h // g].T / math.sqrt(d)
        S[np.triu_indices(L, 1)] = -np.inf
        np.testing.assert_allclose(lse[h], logsumexp(S, axis=1), rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("L,H,Hkv,d", [(300, 4, 2, 16), (111, 2, 1, 8)])
def test_multi_block_core_backward_matches_torch_autograd(small_blocks, L, H, Hkv, d):
    rng = np.random.default_rng(22)
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    do = rng.standard_normal((L, H, d))
    o, lse = orc.attention_core_fwd(q, k, v)
    dq, dk, dv = orc.attention_core_bwd(q, k, v, o, lse, do)
    g = H // Hkv
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(g, dim=1).permute(1, 0, 2)[None],
        tv.repeat_interleave(g, dim=1).permute(1, 0, 2)[None], is_causal=True)[0].permute(1, 0, 2)
    (to * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_multi_block_results_equal_single_block(monkeypatch):
    """Blocked and unblocked runs of every streamed function agree, in both
    precision modes, including the sampled-row helpers at scattered rows."""
    rng = np.random.default_rng(23)
    L, H, Hkv, d = 257, 4, 1, 16
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, Hkv, d))
    v = rng.standard_normal((L, Hkv, d))
    do = rng.standard_normal((L, H, d))
    rows = np.array([0, 3, 40, 41, 128, 200, 256])
    sc = 1 / math.sqrt(d)

    def run(bf):
        o, lse = orc.attention_core_fwd(q, k, v, p_bf16=bf)
        grads = orc.attention_core_bwd(q, k, v, o, lse, do, bf16_operands=bf)
        ro, rl = orc.attention_head_rows(q[rows, 1], rows, k[:, 0], v[:, 0], sc, p_bf16=bf)
        rdq = orc.attention_dq_rows(q[rows, 1], rows, k[:, 0], v[:, 0], do[rows, 1], o[rows, 1], lse[1, rows], sc,
                                    bf16_operands=bf)
        return (o, lse, *grads, ro, rl, rdq)

    for bf in (False, True):
        monkeypatch.setattr(orc, "ROW_BLOCK", None)
        one = run(bf)
        monkeypatch.setattr(orc, "ROW_BLOCK", 5)
        many = run(bf)
        for a_, b_ in zip(one, many):
            np.testing.assert_allclose(b_, a_, rtol=1e-12, atol=1e-12)


def test_default_blocking_streams_long_sequences():
    """Without an override, a long sequence is split into several blocks of
    at most 8 Mi scores each (the branch the multi-block pins exercise)."""
    assert orc.ROW_BLOCK is None
    assert orc._row_block(1 << 20, 1 << 20) == 8
    assert orc._row_block(131072, 131072) == 64
    assert orc._row_block(300, 300) == 300
