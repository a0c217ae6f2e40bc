"""GPU parity of the attention core (no projection, no RoPE) against the
fp64 oracle, through the C ABI, plus bit-exactness across chunk sizes.  The
bound applies against the oracle's precision-model mode (P and dS enter
their products as bf16); the plain fp64 definition is compared as well
(tests/tolerance.py)."""

import math

import numpy as np
import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from oracle import upipe_oracle as orc
from tests.gpu_common import dev, ensure_lib, f64, status_ok
from tests.tolerance import assert_close, assert_close_plain

pytestmark = pytest.mark.gpu

CASES = [
    # L, H, Hkv, U   (ragged tails, one tile, several tiles, U < g and U >= g)
    (1, 1, 1, 1),
    (127, 2, 1, 1),
    (128, 4, 1, 2),
    (129, 4, 2, 2),
    (300, 4, 1, 4),
    (1000, 4, 1, 1),
    (2048, 8, 2, 8),
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _core(L, H, Hkv, U):
    q, k, v, do = synth.core_inputs(L, H, Hkv)
    cfg = upipe.Config(L=L, H=H, Hkv=Hkv, U=U)
    qd, kd, vd, dod = dev(q, k, v, do)
    o, lse = upipe.core_forward(cfg, qd, kd, vd)
    dq, dk, dv = upipe.core_backward(cfg, qd, kd, vd, o, lse, dod)
    torch.cuda.synchronize()
    status_ok()
    return (q, k, v, do), (o, lse, dq, dk, dv)


@pytest.mark.parametrize("L,H,Hkv,U", CASES)
def test_core_fwd_bwd_matches_oracle(L, H, Hkv, U):
    (q, k, v, do), (o, lse, dq, dk, dv) = _core(L, H, Hkv, U)
    q, k, v, do = f64(q), f64(k), f64(v), f64(do)
    got = [f64(t) for t in (o, lse, dq, dk, dv)]
    ro, rlse = orc.attention_core_fwd(q, k, v)  # the forward output: P exact
    # o enters the backward as the bf16 tensor the forward returns
    model = (ro, rlse, *orc.attention_core_bwd(q, k, v, orc.bf16_round(ro), rlse, do, bf16_operands=True))
    po, plse = orc.attention_core_fwd(q, k, v)
    plain = (po, plse, *orc.attention_core_bwd(q, k, v, po, plse, do))
    for g_, m, p, n in zip(got, model, plain, ("o", "lse", "dq", "dk", "dv")):
        assert_close(g_, m, n)
        assert_close_plain(g_, p, m, n)


@pytest.mark.parametrize("L,H,Hkv", [(777, 8, 2), (256, 4, 1)])
def test_core_bit_exact_across_chunk_sizes(L, H, Hkv):
    g = H // Hkv
    Us = [u for u in range(1, H + 1) if H % u == 0 and (u % g == 0 or g % u == 0)]
    ref = None
    for U in Us:
        _, outs = _core(L, H, Hkv, U)
        if ref is None:
            ref = outs
            continue
        for a, b, n in zip(ref, outs, ("o", "lse", "dq", "dk", "dv")):
            assert torch.equal(a, b), f"U={U}: {n} differs from U={Us[0]}"
