"""The per-chunk head exchange of Untied Ulysses across P ranks: the
exchange plan, the packing of the all-to-all buffers, and the chunk loop
that runs the attention core between the exchanges (forward and backward,
over torch.distributed all-to-alls).

"Untied Ulysses Pushes Llama-3-8B Training to 5 Million Tokens" (talk
write-up), paragraph on DeepSpeed Ulysses: activations arrive sharded by
sequence and an all-to-all re-shards Q/K/V by heads before attention (and O
back after it); paragraph on multi-query / grouped-query attention: the
method issues that exchange per head chunk and decouples the exchange of
keys and values from the queries.

Layout: rank r holds sequence rows [r L/P, (r+1) L/P).  Chunk c covers query
heads [c U P, (c+1) U P); rank r owns the U heads c U P + r U .. + U - 1 and
runs their attention over the full sequence, reading KV head h // g for
query head h (g = H / Hkv).  A chunk exchanges K/V only when the KV heads its
ranks need differ from the previous chunk's (at U < g a KV head serves
several chunks).

The chunk loop takes the attention core as two callables, so that it runs
this library's kernels (`gpu_core`) on GPUs with NCCL and any other exact
core on CPU ranks with gloo.  Every run in this repository has one GPU, so
the NCCL path itself is not exercised here.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class ChunkPlan:
    c: int
    q_heads: tuple   # per rank: its U query heads in this chunk
    kv_heads: tuple  # per rank: the KV heads those query heads read
    kv_new: bool     # the chunk needs a K/V exchange (first chunk, or new KV heads)


def plan(H: int, Hkv: int, U: int, P: int) -> list:
    """The chunks of one layer on P ranks with U query heads per rank and chunk."""
    if H % Hkv or H % (U * P):
        raise ValueError("need H % Hkv == 0 and H % (U * P) == 0")
    g = H // Hkv
    if U % g and g % U:
        raise ValueError("U must be a multiple or a divisor of H / Hkv")
    out, prev = [], None
    for c in range(H // (U * P)):
        q = tuple(tuple(range(c * U * P + r * U, c * U * P + (r + 1) * U)) for r in range(P))
        kv = tuple(tuple(sorted({h // g for h in hs})) for hs in q)
        out.append(ChunkPlan(c, q, kv, kv != prev))
        prev = kv
    return out


def rows_of(L: int, P: int, r: int) -> range:
    """Sequence rows rank r holds."""
    if L % P:
        raise ValueError("L must be a multiple of P")
    n = L // P
    return range(r * n, (r + 1) * n)


def pack_heads(local, heads_per_rank):
    """Send buffer of a sequence-to-heads exchange: local [n, heads, d] rows
    of this rank, grouped by destination rank -> [P, n, u, d] (contiguous;
    block s goes to rank s).  heads_per_rank[s] indexes the local head axis."""
    import torch
    return torch.stack([local[:, list(hs)] for hs in heads_per_rank]).contiguous()


def unpack_sequence(recv):
    """Receive buffer of a sequence-to-heads exchange, [P (source rank), n,
    u, d] -> the full sequence of this rank's heads [P n, u, d] (source rank
    order is row order)."""
    return recv.reshape(-1, *recv.shape[2:])


def pack_rows(full, P: int):
    """Send buffer of the heads-to-sequence exchange of O: this rank's heads
    over the full sequence [L, u, d] -> [P, L / P, u, d] (block s holds rank
    s's rows)."""
    return full.reshape(P, full.shape[0] // P, *full.shape[1:]).contiguous()


def unpack_heads(recv):
    """Receive buffer of the heads-to-sequence exchange, [P (source rank),
    n, u, d] -> this rank's rows of every head of the chunk [n, P u, d], heads
    in rank order (= ascending head index within the chunk)."""
    P, n, u, d = recv.shape
    return recv.permute(1, 0, 2, 3).reshape(n, P * u, d)


# ---------------------------------------------------------------- chunk loop

def _exchange(x, group):
    """One all-to-all of a packed [P, ...] buffer: block s goes to rank s;
    returns [P, ...] with block r from rank r."""
    import torch
    import torch.distributed as dist
    out = torch.empty_like(x)
    dist.all_to_all_single(out, x.contiguous(), group=group)
    return out


def forward(q, k, v, H, Hkv, U, core_fwd, group=None):
    """Attention of this rank's sequence shard q [n, H, d], k, v [n, Hkv, d]
    (n = L / P rows, ranks in sequence order).  Per chunk: Q (and K/V when
    the chunk's KV heads change) go from sequence to heads, the rank runs
    core_fwd(q [L, U, d], k, v [L, kv, d]) -> (o [L, U, d], lse [U, L]) on
    its U heads over the whole sequence, and O comes back to sequence shards.
    Returns (o [n, H, d], lse) with lse[c] the [U, L] LSE of this rank's
    heads in chunk c (kept by the head owner for the backward)."""
    import torch
    import torch.distributed as dist
    P = dist.get_world_size(group)
    r = dist.get_rank(group)
    o = torch.empty_like(q)
    lse, kv = {}, None
    for c in plan(H, Hkv, U, P):
        qf = unpack_sequence(_exchange(pack_heads(q, c.q_heads), group))
        if c.kv_new:
            kv = tuple(unpack_sequence(_exchange(pack_heads(t, c.kv_heads), group)) for t in (k, v))
        o_c, lse[c.c] = core_fwd(qf.contiguous(), kv[0].contiguous(), kv[1].contiguous())
        heads = [h for hs in c.q_heads for h in hs]
        o[:, heads] = unpack_heads(_exchange(pack_rows(o_c, P), group))
    return o, lse


def backward(q, k, v, o, lse, do, H, Hkv, U, core_bwd, group=None):
    """Gradients of this rank's shards: dq [n, H, d], dk, dv [n, Hkv, d]
    (sums in fp32, or the shards' dtype if wider; see below).  Per chunk: Q, O, dO (and K/V when they change)
    go from sequence to heads, core_bwd(q, k, v, o, lse, do) -> (dq, dk, dv)
    runs on this rank's heads, dQ comes back to sequence shards, and dK/dV
    come back to the sequence shards of their KV heads, where the partials
    of ranks (U < g: several ranks' query heads read one KV head) and of
    chunks (U < g: a KV head serves several chunks) are summed in fp32."""
    import torch
    import torch.distributed as dist
    P = dist.get_world_size(group)
    dq = torch.empty_like(do)
    acc_t = torch.promote_types(k.dtype, torch.float32)  # fp32 for bf16 shards, wider inputs keep theirs
    dk = torch.zeros(k.shape, dtype=acc_t, device=k.device)
    dv = torch.zeros(v.shape, dtype=acc_t, device=v.device)
    kv = None
    for c in plan(H, Hkv, U, P):
        qf, of, dof = (unpack_sequence(_exchange(pack_heads(t, c.q_heads), group)).contiguous() for t in (q, o, do))
        if c.kv_new:
            kv = tuple(unpack_sequence(_exchange(pack_heads(t, c.kv_heads), group)).contiguous() for t in (k, v))
        dq_c, dk_c, dv_c = core_bwd(qf, kv[0], kv[1], of, lse[c.c], dof)
        heads = [h for hs in c.q_heads for h in hs]
        dq[:, heads] = unpack_heads(_exchange(pack_rows(dq_c, P), group))
        kv_heads = [h for hs in c.kv_heads for h in hs]
        for acc, part in ((dk, dk_c), (dv, dv_c)):
            back = unpack_heads(_exchange(pack_rows(part, P), group)).to(acc_t)
            for j, h in enumerate(kv_heads):
                acc[:, h] += back[:, j]
    return dq, dk, dv


def gpu_core():
    """The attention core of this library as (core_fwd, core_bwd) for
    forward / backward: each call runs upipe_attn_core_fwd / _bwd on the
    current CUDA device over all the heads it is given (one chunk)."""
    from headwise_chunked_context_gb300 import upipe

    def cfg(q, k):
        L, h, _ = q.shape
        return upipe.Config(L=L, H=h, Hkv=k.shape[1], U=h)

    def core_fwd(q, k, v):
        return upipe.core_forward(cfg(q, k), q, k, v)

    def core_bwd(q, k, v, o, lse, do):
        return upipe.core_backward(cfg(q, k), q, k, v, o, lse, do)

    return core_fwd, core_bwd
