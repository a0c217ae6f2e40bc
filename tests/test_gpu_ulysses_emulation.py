"""Untied Ulysses across P ranks, emulated on one GPU: the exchange plan of
headwise_chunked_context_gb300/untied_ulysses.py moves sequence-sharded
Q/K/V/dO to head-sharded full-sequence chunks and O/dQ/dK/dV back, with
the all-to-alls replaced by tensor permutations on the device (no
collective, no kernel waits on another); each emulated rank runs this
library's attention core on its own heads.  The composition must return
the single-GPU core's bits: every head's attention is computed by the same
kernels over the same full-sequence inputs.  (U < g, where two ranks'
query heads share a KV head, sums dK/dV partials across ranks and is
checked within the tolerance instead.)"""

import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from headwise_chunked_context_gb300 import untied_ulysses as uu
from tests.gpu_common import ensure_lib, f64, status_ok
from tests.tolerance import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _all_to_all(sends):
    """sends[r]: rank r's send buffer [P, ...] (block s for rank s) ->
    recvs[s]: [P, ...] (block r from rank r)."""
    P = len(sends)
    return [torch.stack([sends[r][s] for r in range(P)]) for s in range(P)]


def _emulate(L, H, Hkv, U, P):
    q, k, v, do = (t.to("cuda:0") for t in synth.core_inputs(L, H, Hkv))
    rows = [list(uu.rows_of(L, P, r)) for r in range(P)]
    shard = lambda t: [t[rw] for rw in rows]  # sequence shards of each rank
    qs, ks, vs, dos = shard(q), shard(k), shard(v), shard(do)
    o = torch.empty_like(q)
    lse = torch.empty((H, L), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.zeros(k.shape, dtype=torch.float32, device=q.device)
    dv = torch.zeros(v.shape, dtype=torch.float32, device=q.device)
    kv_full = None
    for c in uu.plan(H, Hkv, U, P):
        # sequence -> heads
        qf = [uu.unpack_sequence(b) for b in _all_to_all([uu.pack_heads(qs[r], c.q_heads) for r in range(P)])]
        dof = [uu.unpack_sequence(b) for b in _all_to_all([uu.pack_heads(dos[r], c.q_heads) for r in range(P)])]
        if c.kv_new:
            kf = [uu.unpack_sequence(b) for b in _all_to_all([uu.pack_heads(ks[r], c.kv_heads) for r in range(P)])]
            vf = [uu.unpack_sequence(b) for b in _all_to_all([uu.pack_heads(vs[r], c.kv_heads) for r in range(P)])]
            kv_full = (kf, vf)
        kf, vf = kv_full
        # each rank: the attention core over the full sequence of its heads
        outs = []
        for s in range(P):
            hq, hkv = len(c.q_heads[s]), len(c.kv_heads[s])
            cfg = upipe.Config(L=L, H=hq, Hkv=hkv, U=hq)
            qq, kk, vv, dd = (t.contiguous() for t in (qf[s], kf[s], vf[s], dof[s]))
            o_s, lse_s = upipe.core_forward(cfg, qq, kk, vv)
            dq_s, dk_s, dv_s = upipe.core_backward(cfg, qq, kk, vv, o_s, lse_s, dd)
            outs.append((o_s, lse_s, dq_s, dk_s, dv_s))
        # heads -> sequence for O and dQ; LSE and dK/dV gathered per head
        for name, idx, dst in (("o", 0, o), ("dq", 2, dq)):
            back = _all_to_all([uu.pack_rows(outs[s][idx], P) for s in range(P)])
            heads = [h for hs in c.q_heads for h in hs]
            for r in range(P):
                dst[rows[r][0]:rows[r][-1] + 1, heads] = uu.unpack_heads(back[r])
        for s in range(P):
            lse[list(c.q_heads[s])] = outs[s][1]
            dk[:, list(c.kv_heads[s])] += outs[s][3].float()
            dv[:, list(c.kv_heads[s])] += outs[s][4].float()
    torch.cuda.synchronize()
    status_ok()
    cfg = upipe.Config(L=L, H=H, Hkv=Hkv, U=H)
    ro, rlse = upipe.core_forward(cfg, q, k, v)
    rdq, rdk, rdv = upipe.core_backward(cfg, q, k, v, ro, rlse, do)
    torch.cuda.synchronize()
    status_ok()
    return (o, lse, dq, dk, dv), (ro, rlse, rdq, rdk, rdv)


@pytest.mark.parametrize("L,H,Hkv,U,P", [(1024, 8, 2, 4, 2), (768, 16, 4, 4, 2), (512, 16, 2, 8, 2),
                                         (640, 16, 4, 4, 4)])
def test_emulated_ranks_return_the_single_gpu_bits(L, H, Hkv, U, P):
    """U >= g: every rank holds whole KV groups, so nothing is summed
    across ranks and all five results are identical."""
    (o, lse, dq, dk, dv), (ro, rlse, rdq, rdk, rdv) = _emulate(L, H, Hkv, U, P)
    assert torch.equal(o, ro) and torch.equal(lse, rlse) and torch.equal(dq, rdq)
    assert torch.equal(dk.bfloat16(), rdk) and torch.equal(dv.bfloat16(), rdv)


def test_emulated_ranks_sharing_a_kv_head():
    """U < g: two ranks' query heads read one KV head; O, LSE and dQ are
    still identical, dK/dV are the sum of the ranks' bf16 partials."""
    (o, lse, dq, dk, dv), (ro, rlse, rdq, rdk, rdv) = _emulate(1024, 8, 2, 2, 2)
    assert torch.equal(o, ro) and torch.equal(lse, rlse) and torch.equal(dq, rdq)
    assert_close(f64(dk), f64(rdk), "dk (summed across ranks)")
    assert_close(f64(dv), f64(rdv), "dv (summed across ranks)")


@pytest.mark.parametrize("L,H,Hkv,U", [(1024, 8, 2, 4), (640, 16, 4, 8), (512, 8, 2, 2)])
def test_chunk_loop_with_the_gpu_core_on_one_nccl_rank(L, H, Hkv, U):
    """untied_ulysses.forward / backward with this library's kernels as the
    core, over NCCL with a world of one rank (each all-to-all is a copy):
    the chunk loop returns the single-GPU core's O, LSE and dQ bits, and dK
    / dV within the tolerance (U < g sums a KV head's chunk partials in
    fp32) or bit for bit (U >= g)."""
    import os
    import socket
    import torch.distributed as dist
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda:0"))
    try:
        q, k, v, do = (t.to("cuda:0") for t in synth.core_inputs(L, H, Hkv))
        core_fwd, core_bwd = uu.gpu_core()
        o, lse = uu.forward(q, k, v, H, Hkv, U, core_fwd)
        dq, dk, dv = uu.backward(q, k, v, o, lse, do, H, Hkv, U, core_bwd)
        torch.cuda.synchronize()
        status_ok()
        cfg = upipe.Config(L=L, H=H, Hkv=Hkv, U=U)
        ro, rlse = upipe.core_forward(cfg, q, k, v)
        rdq, rdk, rdv = upipe.core_backward(cfg, q, k, v, ro, rlse, do)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(dq, rdq)
        for c in uu.plan(H, Hkv, U, 1):
            assert torch.equal(lse[c.c], rlse[list(c.q_heads[0])])
        if U >= H // Hkv:
            assert torch.equal(dk.bfloat16(), rdk) and torch.equal(dv.bfloat16(), rdv)
        else:
            assert_close(f64(dk), f64(rdk), "dk (chunk partials summed in fp32)")
            assert_close(f64(dv), f64(rdv), "dv (chunk partials summed in fp32)")
    finally:
        dist.destroy_process_group()
