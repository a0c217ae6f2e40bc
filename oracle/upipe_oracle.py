"""fp64 CPU oracle for the head-chunked GQA/RoPE causal attention layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: it is used by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.
It shares no code with the CUDA path (no kernels, headers, tables or
helpers); both sides only share the seeded input generator, which holds
none of the method's arithmetic.

What it computes, and where that is stated
------------------------------------------
"Untied Ulysses Pushes Llama-3-8B Training to 5 Million Tokens" (orply.com
talk write-up), paragraph on intermediate buffers: the method computes one
group of heads at a time, stores a partial result and reuses the buffers; it
is "not a new attention formula, but a different memory schedule".  So the
oracle is the plain definition of one GQA/RoPE attention layer:

* projections: Q, K, V are "the query, key, and value matrices in the
  transformer layer" (same write-up, Q&A paragraph);  ``QKV = x Wqkv^T``;
* rotary position embedding, RoFormer (listed under "Builds on" on the
  "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
  Chunking" index page);
* exact causal softmax attention per query head, grouped-query mapping
  (the write-up's paragraph on multi-query / grouped-query attention);
* output projection ``out = concat_h(O_h) Wo^T``;
* backward: the exact gradient of ``sum(out * dout)`` via the closed-form
  softmax backward.

Readings of points the pages leave open:

* RoPE pairs (i, i + d/2) ("rotate-half"), angle p * theta^(-2i/d) in fp64,
  rotation by +angle; no frequency scaling.
* scale 1/sqrt(d); no soft-cap, dropout or bias.
* causal mask: key j visible to query i iff j <= i (one sequence).
* GQA: query head h reads KV head h // g, g = H / Hkv.
* LSE: natural log of sum_j exp(scaled score), layout [H, L].
* Wqkv rows: q heads 0..H-1, then k heads, then v heads, d rows each.

Every function below is plain: library matmuls and elementwise NumPy, no
blocking beyond streaming query rows against the full K/V (which changes no
arithmetic that matters at fp64), no fusion.

Precision model ("bf16 in / fp32 accumulate", the stated tolerance's
precision).  By default everything is exact fp64.  With
``bf16_operands=True`` every input of every contraction of the definition is
rounded to the nearest bfloat16 (``bf16_round``) -- that is what "bf16 in"
says -- while every product, sum and element-wise step stays exact fp64
(better than the fp32 the model allows):

* stored tensors that feed the next contraction: Q and K after RoPE, V, the
  attention output O, and dO = dout Wo;
* the softmax tiles of the backward where they enter a product: the
  probabilities P = exp(S - LSE) in P^T dO and in the recomputation of
  O = P V from the forward's LSE, and dS = P * (dP - Delta) in dS K and
  dS^T Q.  P inside dS's element-wise formula is not a contraction input and
  stays exact.

The forward output's own P V (``layer_fwd``) keeps P exact: an online
softmax rounds exp(S - running maximum), a quantity the definition does not
fix, so its rounding is left to the implementation's tolerance.  The
backward recomputes O "from LSE", where P = exp(S - LSE) is the definition's
own quantity (``p_bf16`` of the forward helpers selects this).

This isolates an implementation's own arithmetic (accumulation order, fp32
element-wise math) from the rounding the precision model itself implies.
"""

from __future__ import annotations

import numpy as np

F64 = np.float64


def bf16_round(a) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of ``a``, returned as fp64.

    The value is first rounded to fp32 (as an fp32 accumulator holds it),
    then its fp32 bit pattern is rounded to the upper 16 bits.
    """
    a32 = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = a32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(F64)


# ---------------------------------------------------------------------------
# Rotary position embedding (RoFormer, listed under "Builds on" on the
# "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
# Chunking" index page).  Rotate-half pairing is a reading: the pages are
# silent on it.
# ---------------------------------------------------------------------------

def rope_angles(positions, d: int, theta: float) -> np.ndarray:
    """Angles [n, d/2] in fp64: angle[p, i] = p * theta^(-2i/d)."""
    positions = np.asarray(positions, dtype=F64)
    i = np.arange(d // 2, dtype=F64)
    inv_freq = np.power(F64(theta), -2.0 * i / d)
    return np.outer(positions, inv_freq)


def rope_apply(x: np.ndarray, positions, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate each head vector of ``x`` [n, nh, d] at its position.

    Pair (a, b) = (x[..., i], x[..., i + d/2]) maps to
    (a cos t - b sin t, a sin t + b cos t); ``inverse`` rotates by -t,
    which is the transpose of the forward rotation (used for gradients).
    """
    n, nh, d = x.shape
    ang = rope_angles(positions, d, theta)  # [n, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    if inverse:
        s = -s
    a = x[..., : d // 2]
    b = x[..., d // 2:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


# ---------------------------------------------------------------------------
# Projections.  Wqkv rows are [q heads | k heads | v heads], d rows each.
# ---------------------------------------------------------------------------

def split_qkv(qkv: np.ndarray, H: int, Hkv: int, d: int):
    L = qkv.shape[0]
    q = qkv[:, : H * d].reshape(L, H, d)
    k = qkv[:, H * d: (H + Hkv) * d].reshape(L, Hkv, d)
    v = qkv[:, (H + Hkv) * d:].reshape(L, Hkv, d)
    return q, k, v


def project_qkv(x, Wqkv, H, Hkv, d, theta, rope=True):
    """Q, K, V [L, heads, d] after the projection and (optionally) RoPE."""
    x = np.asarray(x, dtype=F64)
    qkv = x @ np.asarray(Wqkv, dtype=F64).T
    q, k, v = split_qkv(qkv, H, Hkv, d)
    if rope:
        pos = np.arange(x.shape[0])
        q = rope_apply(q, pos, theta)
        k = rope_apply(k, pos, theta)
    return q, k, v


# ---------------------------------------------------------------------------
# Exact causal attention, one query head at a time.
# ---------------------------------------------------------------------------

# Query rows per streamed block.  None sizes blocks so that one block's
# score matrix stays near 64 MB; tests set a small value to run the
# multi-block path on small inputs.
ROW_BLOCK = None


def _row_block(n: int, L: int) -> int:
    if ROW_BLOCK is not None:
        return max(1, min(n, int(ROW_BLOCK)))
    return max(1, min(n, (8 << 20) // max(L, 1)))


def _op(a, bf16_operands):
    """A contraction input under the precision model (module header)."""
    return bf16_round(a) if bf16_operands else a


def attention_head_rows(qr, qpos, k, v, scale, p_bf16=False):
    """O rows and LSE for query rows ``qr`` [n, d] at positions ``qpos``.

    ``k``, ``v`` [Lk, d] are this head's keys/values (KV head h // g).
    Key j is visible to the query at position p iff j <= p.  With ``p_bf16``
    the probabilities exp(S - LSE) enter P V as bf16 (O recomputed from the
    LSE, module header).
    """
    qr = np.asarray(qr, dtype=F64)
    qpos = np.asarray(qpos)
    n = qr.shape[0]
    o = np.zeros((n, v.shape[1]), dtype=F64)
    lse = np.zeros(n, dtype=F64)
    bs = _row_block(n, k.shape[0])
    for s0 in range(0, n, bs):
        s1 = min(n, s0 + bs)
        top = int(qpos[s0:s1].max()) + 1
        S = (qr[s0:s1] @ k[:top].T) * scale
        mask = np.arange(top)[None, :] > qpos[s0:s1, None]
        S[mask] = -np.inf
        m = S.max(axis=1)
        l = np.exp(S - m[:, None]).sum(axis=1)
        lse[s0:s1] = m + np.log(l)
        P = np.exp(S - lse[s0:s1, None])
        o[s0:s1] = _op(P, p_bf16) @ v[:top]
    return o, lse


def attention_core_fwd(q, k, v, causal=True, p_bf16=False):
    """O [L, H, d] and LSE [H, L] for q [L, H, d], k/v [L, Hkv, d]; with
    ``p_bf16`` P enters P V as bf16 (see attention_head_rows)."""
    assert causal, "only the causal square mask is defined here"
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    L, H, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    scale = 1.0 / np.sqrt(d)
    o = np.zeros_like(q)
    lse = np.zeros((H, L), dtype=F64)
    pos = np.arange(L)
    for h in range(H):
        o[:, h], lse[h] = attention_head_rows(q[:, h], pos, k[:, h // g], v[:, h // g], scale, p_bf16)
    return o, lse


def attention_core_bwd(q, k, v, o, lse, do, bf16_operands=False):
    """dq, dk, dv for the causal core, closed-form softmax backward.

    P = exp(S - LSE), dV = P^T dO, dP = dO V^T, Delta = rowsum(dO * O),
    dS = P * (dP - Delta), dQ = dS K * scale, dK = dS^T Q * scale.
    dK/dV of a KV head sum over the g query heads that read it.  With
    ``bf16_operands`` P (in P^T dO) and dS (in dS K, dS^T Q) enter their
    products as bf16.
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    o = np.asarray(o, dtype=F64)
    do = np.asarray(do, dtype=F64)
    lse = np.asarray(lse, dtype=F64)
    L, H, d = q.shape
    Hkv = k.shape[1]
    g = H // Hkv
    scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    bs = _row_block(L, L)
    for h in range(H):
        kh, vh = k[:, h // g], v[:, h // g]
        delta = np.sum(do[:, h] * o[:, h], axis=1)
        for s0 in range(0, L, bs):
            s1 = min(L, s0 + bs)
            top = s1
            S = (q[s0:s1, h] @ kh[:top].T) * scale
            mask = np.arange(top)[None, :] > np.arange(s0, s1)[:, None]
            P = np.exp(S - lse[h, s0:s1, None])
            P[mask] = 0.0
            dv[:top, h // g] += _op(P, bf16_operands).T @ do[s0:s1, h]
            dP = do[s0:s1, h] @ vh[:top].T
            dS = _op(P * (dP - delta[s0:s1, None]), bf16_operands)
            dq[s0:s1, h] = (dS @ kh[:top]) * scale
            dk[:top, h // g] += (dS.T @ q[s0:s1, h]) * scale
    return dq, dk, dv


def attention_dq_rows(qr, qpos, k, v, dor, orow, lser, scale, bf16_operands=False):
    """dQ rows for sampled query rows of one head (needs only that row's
    O, dO and LSE: Delta_i = sum_k dO_ik O_ik)."""
    qr = np.asarray(qr, dtype=F64)
    dor = np.asarray(dor, dtype=F64)
    orow = np.asarray(orow, dtype=F64)
    qpos = np.asarray(qpos)
    n = qr.shape[0]
    dq = np.zeros_like(qr)
    bs = _row_block(n, k.shape[0])
    for s0 in range(0, n, bs):
        s1 = min(n, s0 + bs)
        top = int(qpos[s0:s1].max()) + 1
        S = (qr[s0:s1] @ k[:top].T) * scale
        mask = np.arange(top)[None, :] > qpos[s0:s1, None]
        P = np.exp(S - np.asarray(lser[s0:s1], dtype=F64)[:, None])
        P[mask] = 0.0
        delta = np.sum(dor[s0:s1] * orow[s0:s1], axis=1)
        dP = dor[s0:s1] @ v[:top].T
        dq[s0:s1] = (_op(P * (dP - delta[:, None]), bf16_operands) @ k[:top]) * scale
    return dq


def attention_dkv_tail(q_tail, k_tail, v_tail, do_tail, o_tail, lse_tail, scale, bf16_operands=False):
    """dK, dV of the last T keys of one head pair, from the last T queries.

    Under the causal mask only queries at or after a key's position reach
    it, so the last T keys see exactly the last T queries: this is the
    full gradient for those keys.  Arrays are [T, d] (LSE [T]).
    """
    q_tail = np.asarray(q_tail, dtype=F64)
    k_tail = np.asarray(k_tail, dtype=F64)
    v_tail = np.asarray(v_tail, dtype=F64)
    do_tail = np.asarray(do_tail, dtype=F64)
    o_tail = np.asarray(o_tail, dtype=F64)
    T = q_tail.shape[0]
    S = (q_tail @ k_tail.T) * scale
    mask = np.arange(T)[None, :] > np.arange(T)[:, None]
    P = np.exp(S - np.asarray(lse_tail, dtype=F64)[:, None])
    P[mask] = 0.0
    delta = np.sum(do_tail * o_tail, axis=1)
    dP = do_tail @ v_tail.T
    dS = _op(P * (dP - delta[:, None]), bf16_operands)
    return (dS.T @ q_tail) * scale, _op(P, bf16_operands).T @ do_tail


# ---------------------------------------------------------------------------
# The layer: plain (all heads at once) definition.
# ---------------------------------------------------------------------------

def layer_fwd(x, Wqkv, Wo, H, Hkv, theta, d=None, bf16_operands=False):
    """out [L, D], LSE [H, L], O [L, H, d] of one GQA/RoPE attention layer."""
    x = np.asarray(x, dtype=F64)
    Wo = np.asarray(Wo, dtype=F64)
    if d is None:
        d = Wo.shape[1] // H
    q, k, v = project_qkv(x, Wqkv, H, Hkv, d, theta)
    q, k, v = _op(q, bf16_operands), _op(k, bf16_operands), _op(v, bf16_operands)
    o, lse = attention_core_fwd(q, k, v)  # the forward's own P V: P exact (module header)
    o = _op(o, bf16_operands)
    out = o.reshape(x.shape[0], H * d) @ Wo.T
    return out, lse, o


def layer_bwd(x, Wqkv, Wo, dout, H, Hkv, theta, d=None, bf16_operands=False, kept_o=False):
    """dx [L, D], dWqkv [(H+2Hkv)d, D], dWo [D, H d]: gradient of sum(out*dout).

    With ``bf16_operands`` every contraction input is rounded to bf16 (see
    the module header); the rounding itself is treated as the identity in
    the chain rule.  ``kept_o`` selects the O the backward reads under that
    model: False, O recomputed from the forward's LSE (P enters P V as
    bf16); True, the forward's own output kept from the forward pass (its
    P V keeps P exact, as in layer_fwd).  Without ``bf16_operands`` the two
    are the same exact O.
    """
    x = np.asarray(x, dtype=F64)
    Wqkv = np.asarray(Wqkv, dtype=F64)
    Wo = np.asarray(Wo, dtype=F64)
    dout = np.asarray(dout, dtype=F64)
    L = x.shape[0]
    if d is None:
        d = Wo.shape[1] // H
    q, k, v = project_qkv(x, Wqkv, H, Hkv, d, theta)
    q, k, v = _op(q, bf16_operands), _op(k, bf16_operands), _op(v, bf16_operands)
    # O recomputed from the forward's LSE (P = exp(S - LSE), bf16 in P V
    # under the precision model), or the forward's kept output.
    o, lse = attention_core_fwd(q, k, v, p_bf16=bf16_operands and not kept_o)
    o = _op(o, bf16_operands)
    o_flat = o.reshape(L, H * d)
    dWo = dout.T @ o_flat
    do = _op((dout @ Wo).reshape(L, H, d), bf16_operands)
    dq, dk, dv = attention_core_bwd(q, k, v, o, lse, do, bf16_operands=bf16_operands)
    pos = np.arange(L)
    dq = rope_apply(dq, pos, theta, inverse=True)
    dk = rope_apply(dk, pos, theta, inverse=True)
    dqkv = np.concatenate([dq.reshape(L, -1), dk.reshape(L, -1), dv.reshape(L, -1)], axis=1)
    dWqkv = dqkv.T @ x
    dx = dqkv @ Wqkv
    return dx, dWqkv, dWo


# ---------------------------------------------------------------------------
# The layer computed one head-chunk at a time (the write-up's paragraph on
# intermediate buffers: one group of heads per stage, partial result stored,
# buffers reused).  Used only to pin the invariant that every chunk size U
# gives the plain layer's result.
# ---------------------------------------------------------------------------

def chunk_heads(c: int, U: int, H: int, Hkv: int):
    """Query heads and KV heads of chunk c."""
    g = H // Hkv
    qh = list(range(c * U, (c + 1) * U))
    kvh = sorted({h // g for h in qh})
    return qh, kvh


def _w_rows(heads, base, d):
    return np.concatenate([np.arange((base + h) * d, (base + h + 1) * d) for h in heads])


def layer_fwd_chunked(x, Wqkv, Wo, H, Hkv, theta, U, d=None):
    x = np.asarray(x, dtype=F64)
    Wqkv = np.asarray(Wqkv, dtype=F64)
    Wo = np.asarray(Wo, dtype=F64)
    L, D = x.shape
    if d is None:
        d = Wo.shape[1] // H
    g = H // Hkv
    out = np.zeros((L, D), dtype=F64)
    lse = np.zeros((H, L), dtype=F64)
    pos = np.arange(L)
    scale = 1.0 / np.sqrt(d)
    for c in range(H // U):
        qh, kvh = chunk_heads(c, U, H, Hkv)
        q = (x @ Wqkv[_w_rows(qh, 0, d)].T).reshape(L, len(qh), d)
        kk = (x @ Wqkv[_w_rows(kvh, H, d)].T).reshape(L, len(kvh), d)
        vv = (x @ Wqkv[_w_rows(kvh, H + Hkv, d)].T).reshape(L, len(kvh), d)
        q = rope_apply(q, pos, theta)
        kk = rope_apply(kk, pos, theta)
        oc = np.zeros((L, len(qh), d), dtype=F64)
        for j, h in enumerate(qh):
            kv = kvh.index(h // g)
            oc[:, j], lse[h] = attention_head_rows(q[:, j], pos, kk[:, kv], vv[:, kv], scale)
        cols = np.arange(qh[0] * d, (qh[-1] + 1) * d)
        out += oc.reshape(L, -1) @ Wo[:, cols].T
    return out, lse


def layer_bwd_chunked(x, Wqkv, Wo, dout, H, Hkv, theta, U, d=None):
    x = np.asarray(x, dtype=F64)
    Wqkv = np.asarray(Wqkv, dtype=F64)
    Wo = np.asarray(Wo, dtype=F64)
    dout = np.asarray(dout, dtype=F64)
    L, D = x.shape
    if d is None:
        d = Wo.shape[1] // H
    g = H // Hkv
    pos = np.arange(L)
    dx = np.zeros((L, D), dtype=F64)
    dWqkv = np.zeros_like(Wqkv)
    dWo = np.zeros_like(Wo)
    for c in range(H // U):
        qh, kvh = chunk_heads(c, U, H, Hkv)
        q = rope_apply((x @ Wqkv[_w_rows(qh, 0, d)].T).reshape(L, len(qh), d), pos, theta)
        kk = rope_apply((x @ Wqkv[_w_rows(kvh, H, d)].T).reshape(L, len(kvh), d), pos, theta)
        vv = (x @ Wqkv[_w_rows(kvh, H + Hkv, d)].T).reshape(L, len(kvh), d)
        # The chunk's query heads with the KV heads they read form a GQA core
        # of len(qh) query heads over len(kvh) KV heads (one KV head if U < g).
        oc, lsec = attention_core_fwd(q, kk, vv)
        cols = np.arange(qh[0] * d, (qh[-1] + 1) * d)
        dWo[:, cols] = dout.T @ oc.reshape(L, -1)
        doc = (dout @ Wo[:, cols]).reshape(L, len(qh), d)
        dq, dk, dv = attention_core_bwd(q, kk, vv, oc, lsec, doc)
        dq = rope_apply(dq, pos, theta, inverse=True)
        dk = rope_apply(dk, pos, theta, inverse=True)
        rq = _w_rows(qh, 0, d)
        dWqkv[rq] = dq.reshape(L, -1).T @ x
        dx += dq.reshape(L, -1) @ Wqkv[rq]
        rk = _w_rows(kvh, H, d)
        rv = _w_rows(kvh, H + Hkv, d)
        # With U < g several chunks read the same KV head: its gradient is
        # the sum over those chunks.
        dWqkv[rk] += dk.reshape(L, -1).T @ x
        dWqkv[rv] += dv.reshape(L, -1).T @ x
        dx += dk.reshape(L, -1) @ Wqkv[rk] + dv.reshape(L, -1) @ Wqkv[rv]
    return dx, dWqkv, dWo


# ---------------------------------------------------------------------------
# Activation-memory arithmetic of the head-chunked schedule (the write-up's
# paragraph on intermediate buffers: one chunk-sized buffer set, reused).
# ---------------------------------------------------------------------------

def chunk_kv_heads(U: int, H: int, Hkv: int) -> int:
    g = H // Hkv
    return U // g if U >= g else 1


def intermediate_bytes(L: int, U: int, H: int, Hkv: int, d: int, elem: int = 2) -> int:
    """Bytes of one chunk's Q, K, V and O buffers: L*d*elem*(2U + 2 kv_c).

    With U = H this is the unchunked layer's Q/K/V/O; the ratio to it is
    exactly U/H whenever U >= g.
    """
    kvc = chunk_kv_heads(U, H, Hkv)
    return L * d * elem * (2 * U + 2 * kvc)
