"""Index arithmetic of the per-chunk head exchange of Untied Ulysses across
ranks, executed with gloo all-to-alls on CPU (world size 2).  Every rank must
receive exactly its own heads' Q over the full sequence, the K/V heads they
read (exchanged only when they change), and get O back as its sequence rows
of every head of the chunk."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from headwise_chunked_context_gb300 import untied_ulysses as uu


def test_plan_head_ownership_and_kv_reuse():
    p = uu.plan(H=8, Hkv=2, U=1, P=2)  # g = 4: two chunks share each KV head
    assert [c.q_heads for c in p] == [((0,), (1,)), ((2,), (3,)), ((4,), (5,)), ((6,), (7,))]
    assert [c.kv_heads for c in p] == [((0,), (0,)), ((0,), (0,)), ((1,), (1,)), ((1,), (1,))]
    assert [c.kv_new for c in p] == [True, False, True, False]
    p = uu.plan(H=32, Hkv=8, U=8, P=2)  # U = 2 g: each rank reads two KV heads
    assert p[1].q_heads[1] == tuple(range(24, 32)) and p[1].kv_heads[1] == (6, 7)
    assert all(c.kv_new for c in p)
    with pytest.raises(ValueError):
        uu.plan(H=8, Hkv=2, U=3, P=2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, cases, errors):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for L, H, Hkv, U, d in cases:
            g = torch.Generator().manual_seed(7)
            q = torch.randn(L, H, d, generator=g)
            k = torch.randn(L, Hkv, d, generator=g)
            v = torch.randn(L, Hkv, d, generator=g)
            mine = list(uu.rows_of(L, world, rank))
            kv_have = None
            for c in uu.plan(H, Hkv, U, world):
                # Q: my rows of every rank's heads -> the full sequence of mine
                send = uu.pack_heads(q[mine], c.q_heads)
                recv = torch.empty_like(send)
                dist.all_to_all_single(recv, send)
                got = uu.unpack_sequence(recv)
                assert torch.equal(got, q[:, list(c.q_heads[rank])]), (c, "q")
                # K/V only when the chunk's KV heads change
                if c.kv_new:
                    for t, name in ((k, "k"), (v, "v")):
                        send = uu.pack_heads(t[mine], c.kv_heads)
                        recv = torch.empty_like(send)
                        dist.all_to_all_single(recv, send)
                        assert torch.equal(uu.unpack_sequence(recv), t[:, list(c.kv_heads[rank])]), (c, name)
                    kv_have = c.kv_heads[rank]
                assert kv_have == c.kv_heads[rank]
                # O (stand-in: O_h = 2 q_h): heads -> my rows of all heads of the chunk
                o_full = 2 * got
                send = uu.pack_rows(o_full, world)
                recv = torch.empty_like(send)
                dist.all_to_all_single(recv, send)
                heads = [h for hs in c.q_heads for h in hs]
                assert torch.equal(uu.unpack_heads(recv), 2 * q[mine][:, heads]), (c, "o")
    except AssertionError as e:
        errors.put(f"rank {rank}: {e}")
    finally:
        dist.destroy_process_group()


def test_exchange_on_two_gloo_ranks():
    cases = [(64, 8, 2, 1, 4), (64, 8, 2, 2, 4), (32, 8, 2, 4, 8), (96, 16, 4, 2, 4)]
    ctx = mp.get_context("spawn")
    errors = ctx.Queue()
    mp.start_processes(_rank, args=(2, _free_port(), cases, errors), nprocs=2, start_method="spawn")
    msgs = []
    while not errors.empty():
        msgs.append(errors.get())
    assert not msgs, msgs


# ------------------------------------------- chunk loop on gloo ranks (CPU)

def _oracle_core():
    """The fp64 oracle as the attention core (the GPU path passes
    untied_ulysses.gpu_core() instead)."""
    import numpy as np
    from oracle import upipe_oracle as orc

    def core_fwd(q, k, v):
        o, lse = orc.attention_core_fwd(q.numpy(), k.numpy(), v.numpy())
        return torch.from_numpy(o), torch.from_numpy(lse)

    def core_bwd(q, k, v, o, lse, do):
        return tuple(torch.from_numpy(np.ascontiguousarray(t)) for t in
                     orc.attention_core_bwd(q.numpy(), k.numpy(), v.numpy(), o.numpy(), lse.numpy(), do.numpy()))

    return core_fwd, core_bwd


def _loop_rank(rank, world, port, cases, errors):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import upipe_oracle as orc
        core_fwd, core_bwd = _oracle_core()
        for L, H, Hkv, U, d in cases:
            g = torch.Generator().manual_seed(11)
            q, k, v, do = (torch.randn(L, n, d, generator=g, dtype=torch.float64) for n in (H, Hkv, Hkv, H))
            mine = list(uu.rows_of(L, world, rank))
            o, lse = uu.forward(q[mine], k[mine], v[mine], H, Hkv, U, core_fwd)
            dq, dk, dv = uu.backward(q[mine], k[mine], v[mine], o, lse, do[mine], H, Hkv, U, core_bwd)
            ro, rlse = orc.attention_core_fwd(q.numpy(), k.numpy(), v.numpy())
            rdq, rdk, rdv = orc.attention_core_bwd(q.numpy(), k.numpy(), v.numpy(), ro, rlse, do.numpy())
            for name, got, ref in (("o", o, ro), ("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
                err = float((got.double() - torch.from_numpy(ref)[mine]).abs().max())
                assert err < 1e-10, f"{(L, H, Hkv, U)} {name}: max error {err:.3e}"
            for c in uu.plan(H, Hkv, U, world):
                ref = torch.from_numpy(rlse)[list(c.q_heads[rank])]
                assert float((lse[c.c] - ref).abs().max()) < 1e-10, f"{(L, H, Hkv, U)} lse chunk {c.c}"
    except AssertionError as e:
        errors.put(f"rank {rank}: {e}")
    finally:
        dist.destroy_process_group()


def test_chunk_loop_on_two_gloo_ranks_equals_the_single_process_core():
    """The whole Untied Ulysses chunk loop (exchanges, per-rank core, dK/dV
    partials summed on their owners) with the fp64 oracle as the core: every
    rank's shard of O, dQ, dK, dV and its heads' LSE equal the single-process
    attention, for U >= g and U < g (shared KV heads across ranks and chunks)."""
    cases = [(64, 8, 2, 4, 4), (64, 8, 2, 2, 4), (48, 8, 2, 1, 4), (32, 16, 4, 2, 8)]
    ctx = mp.get_context("spawn")
    errors = ctx.Queue()
    mp.start_processes(_loop_rank, args=(2, _free_port(), cases, errors), nprocs=2, start_method="spawn")
    msgs = []
    while not errors.empty():
        msgs.append(errors.get())
    assert not msgs, msgs


def test_plan_and_shards_reject_bad_shapes():
    with pytest.raises(ValueError):
        uu.plan(H=8, Hkv=3, U=1, P=2)   # H % Hkv != 0
    with pytest.raises(ValueError):
        uu.plan(H=8, Hkv=2, U=4, P=4)   # H % (U P) != 0
    with pytest.raises(ValueError):
        uu.rows_of(L=10, P=4, r=0)      # L % P != 0
    assert list(uu.rows_of(L=12, P=4, r=3)) == [9, 10, 11]
    # every query head is owned exactly once across chunks and ranks
    for H, Hkv, U, P in ((64, 8, 8, 8), (32, 8, 1, 4), (16, 16, 2, 2)):
        owned = [h for c in uu.plan(H, Hkv, U, P) for hs in c.q_heads for h in hs]
        assert sorted(owned) == list(range(H))
