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

class _Exchange:
    """One all-to-all of a packed [P, ...] buffer (block s goes to rank s;
    the result holds block r from rank r), issued asynchronously: on NCCL
    it runs on the communicator's stream beside the compute already
    enqueued, and `result()` makes the current stream wait for it."""

    def __init__(self, x, group):
        import torch
        import torch.distributed as dist
        self.out = torch.empty_like(x)
        self.work = dist.all_to_all_single(self.out, x.contiguous(), group=group, async_op=True)

    def result(self):
        self.work.wait()
        return self.out


def _to_heads(x, heads, group):
    return _Exchange(pack_heads(x, heads), group)


def forward(q, k, v, H, Hkv, U, core_fwd, group=None):
    """Attention of this rank's sequence shard q [n, H, d], k, v [n, Hkv, d]
    (n = L / P rows, ranks in sequence order).  Per chunk: Q (and K/V when
    the chunk's KV heads change) go from sequence to heads, the rank runs
    core_fwd(q [L, U, d], k, v [L, kv, d]) -> (o [L, U, d], lse [U, L]) on
    its U heads over the whole sequence, and O comes back to sequence shards.
    The next chunk's exchanges are issued before this chunk's attention, and
    a chunk's O is collected only after the next chunk's attention, so that
    on GPUs the exchanges run beside the attention (at most two chunks'
    exchange buffers live at once: memory stays proportional to U).  Returns (o [n, H, d], lse) with lse[c]
    the [U, L] LSE of this rank's heads in chunk c (kept by the head owner
    for the backward)."""
    import torch
    import torch.distributed as dist
    P = dist.get_world_size(group)
    chunks = plan(H, Hkv, U, P)

    def issue(c):
        kvx = tuple(_to_heads(t, c.kv_heads, group) for t in (k, v)) if c.kv_new else None
        return _to_heads(q, c.q_heads, group), kvx

    o = torch.empty_like(q)

    def land(done):  # O of a finished chunk into this rank's rows
        c, ox = done
        o[:, [h for hs in c.q_heads for h in hs]] = unpack_heads(ox.result())

    lse, kv = {}, None
    pending, back = issue(chunks[0]), None
    for i, c in enumerate(chunks):
        qx, kvx = pending
        if i + 1 < len(chunks):
            pending = issue(chunks[i + 1])
        qf = unpack_sequence(qx.result()).contiguous()
        if kvx is not None:
            kv = tuple(unpack_sequence(x.result()).contiguous() for x in kvx)
        o_c, lse[c.c] = core_fwd(qf, kv[0], kv[1])
        if back is not None:  # the previous chunk's O has had this chunk's attention to arrive
            land(back)
        back = (c, _Exchange(pack_rows(o_c, P), group))
    land(back)
    return o, lse


def backward(q, k, v, o, lse, do, H, Hkv, U, core_bwd, group=None):
    """Gradients of this rank's shards: dq [n, H, d], dk, dv [n, Hkv, d]
    (sums in fp32, or the shards' dtype if wider).  Per chunk: Q, O, dO (and
    K/V when they change) go from sequence to heads, core_bwd(q, k, v, o,
    lse, do) -> (dq, dk, dv) runs on this rank's heads, dQ comes back to
    sequence shards, and dK/dV come back to the sequence shards of their KV
    heads, where the partials of ranks (U < g: several ranks' query heads
    read one KV head) and of chunks (U < g: a KV head serves several chunks)
    are summed.  The next chunk's exchanges are issued before this chunk's
    attention, as in the forward."""
    import torch
    import torch.distributed as dist
    P = dist.get_world_size(group)
    chunks = plan(H, Hkv, U, P)
    acc_t = torch.promote_types(k.dtype, torch.float32)  # fp32 for bf16 shards, wider inputs keep theirs
    dq = torch.empty_like(do)
    dk = torch.zeros(k.shape, dtype=acc_t, device=k.device)
    dv = torch.zeros(v.shape, dtype=acc_t, device=v.device)

    def issue(c):
        kvx = tuple(_to_heads(t, c.kv_heads, group) for t in (k, v)) if c.kv_new else None
        return tuple(_to_heads(t, c.q_heads, group) for t in (q, o, do)), kvx

    def land(done):  # a finished chunk's gradients into this rank's shards
        c, (dqx, dkx, dvx) = done
        dq[:, [h for hs in c.q_heads for h in hs]] = unpack_heads(dqx.result())
        kv_heads = [h for hs in c.kv_heads for h in hs]
        for acc, x in ((dk, dkx), (dv, dvx)):
            part = unpack_heads(x.result()).to(acc_t)
            for j, h in enumerate(kv_heads):
                acc[:, h] += part[:, j]

    kv = None
    pending, back = issue(chunks[0]), None
    for i, c in enumerate(chunks):
        qx, kvx = pending
        if i + 1 < len(chunks):
            pending = issue(chunks[i + 1])
        qf, of, dof = (unpack_sequence(x.result()).contiguous() for x in qx)
        if kvx is not None:
            kv = tuple(unpack_sequence(x.result()).contiguous() for x in kvx)
        dq_c, dk_c, dv_c = core_bwd(qf, kv[0], kv[1], of, lse[c.c], dof)
        if back is not None:
            land(back)
        back = (c, tuple(_Exchange(pack_rows(t, P), group) for t in (dq_c, dk_c, dv_c)))
    land(back)
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
