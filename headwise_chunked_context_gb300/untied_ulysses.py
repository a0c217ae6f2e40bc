"""Index arithmetic of the per-chunk head exchange of Untied Ulysses across P
ranks (host logic only; this library itself runs on one GPU).

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
