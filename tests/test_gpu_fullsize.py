"""GPU parity at the full workload sizes, on outputs the fp64 oracle can
compute one by one, plus bit-exactness of every chunk size U at those sizes.

Sampled checks (oracle fp64 in its bf16-materialisation mode: Q, K, V, O
and dO rounded to bf16 where a bf16 layer stores them; the GPU run is the
full-size run):
 * forward rows: out and LSE of sampled query positions (each needs that
   row's Q and the K/V of every earlier position);
 * backward tail: under the causal mask the last T keys are seen only by the
   last T queries, so dQ, dK, dV -- and hence dx -- of the last T positions
   follow from those T rows alone (plus their O/LSE rows);
 * one head's columns of dWo (needs that head's O for every row).
Everything else at these sizes is pinned by bit-exactness against U = H and
by the small-size full parity tests.
"""

import math

import numpy as np
import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from oracle import upipe_oracle as orc
from tests.gpu_common import ensure_lib, f64, status_ok
from tests.tolerance import assert_close, assert_max_abs

pytestmark = pytest.mark.gpu

D_HEAD = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _rows(L, n=12, seed=0):
    """(uniform rows, edge rows).  The rel-L2 of a tensor is estimated on rows
    drawn uniformly; edge rows (first, tile boundaries, last) are checked
    element-wise only, since they are not a sample of the tensor."""
    rng = np.random.default_rng(seed)
    uni = np.unique(rng.integers(0, L, n)).astype(np.int64)
    edge = np.array(sorted({x for x in (0, 1, 127, 128, 129, L // 2, L - 129, L - 1) if 0 <= x < L}), dtype=np.int64)
    return uni, edge


def _proj_rows(x, W, rows_w, positions, theta, rope):
    """Projection of x[positions] onto Wqkv rows `rows_w` (fp64), RoPE'd."""
    xr = x[positions].to(torch.float64).numpy()
    y = xr @ W[rows_w].to(torch.float64).numpy().T
    n_heads = len(rows_w) // D_HEAD
    y = y.reshape(len(positions), n_heads, D_HEAD)
    return orc.rope_apply(y, positions, theta) if rope else y


def _kv_all(x, W, shape, upto, block=16384):
    """fp64 K (RoPE'd) and V [upto, Hkv, d] from x[:upto], blockwise."""
    H, Hkv = shape.H, shape.Hkv
    rk = np.arange(H * D_HEAD, (H + Hkv) * D_HEAD)
    rv = np.arange((H + Hkv) * D_HEAD, (H + 2 * Hkv) * D_HEAD)
    K = np.empty((upto, Hkv, D_HEAD))
    V = np.empty((upto, Hkv, D_HEAD))
    for s0 in range(0, upto, block):
        pos = np.arange(s0, min(upto, s0 + block))
        K[pos] = _proj_rows(x, W, rk, pos, shape.theta, True)
        V[pos] = _proj_rows(x, W, rv, pos, shape.theta, False)
    return K, V


def _run_layer(shape, U, inputs):
    x, w, wo, dout = inputs
    cfg = upipe.Config(L=shape.L, D=shape.D, H=shape.H, Hkv=shape.Hkv, U=U, rope_theta=shape.theta)
    xd, wd, wod, dd = (t.to("cuda:0") for t in inputs)
    out, lse, _ = upipe.layer_forward(cfg, xd, wd, wod)
    dx, dwqkv, dwo = upipe.layer_backward(cfg, xd, wd, wod, dd, lse)
    torch.cuda.synchronize()
    status_ok()
    res = tuple(t.cpu() for t in (out, lse, dx, dwqkv, dwo))
    del xd, wd, wod, dd, out, lse, dx, dwqkv, dwo
    torch.cuda.empty_cache()
    return res


def _check_layer_rows(shape, inputs, res, fwd_rows, tail, dwo_head=None):
    x, w, wo, dout = inputs
    out, lse, dx, dwqkv, dwo = res
    H, Hkv, L = shape.H, shape.Hkv, shape.L
    g = H // Hkv
    scale = 1 / math.sqrt(D_HEAD)
    wq_rows = np.arange(H * D_HEAD)
    uni, edge = fwd_rows
    fwd_rows = np.unique(np.concatenate([uni, edge]))
    need = L if tail else int(fwd_rows.max()) + 1
    K, V = _kv_all(x, w, shape, need)
    K, V = orc.bf16_round(K), orc.bf16_round(V)
    Wo = wo.to(torch.float64).numpy()

    # forward rows
    Qr = orc.bf16_round(_proj_rows(x, w, wq_rows, fwd_rows, shape.theta, True))
    Or = np.empty((len(fwd_rows), H, D_HEAD))
    Lr = np.empty((H, len(fwd_rows)))
    for h in range(H):
        Or[:, h], Lr[h] = orc.attention_head_rows(Qr[:, h], fwd_rows, K[:, h // g], V[:, h // g], scale)
    ref_out = orc.bf16_round(Or).reshape(len(fwd_rows), -1) @ Wo.T
    iu = np.searchsorted(fwd_rows, uni)
    ie = np.searchsorted(fwd_rows, edge)
    assert_close(f64(out[uni]), ref_out[iu], "out rows")
    assert_close(f64(lse[:, uni]), Lr[:, iu], "lse rows")
    assert_max_abs(f64(out[edge]), ref_out[ie], "out edge rows")
    assert_max_abs(f64(lse[:, edge]), Lr[:, ie], "lse edge rows")

    if tail:
        T = tail
        tpos = np.arange(L - T, L)
        Qt = orc.bf16_round(_proj_rows(x, w, wq_rows, tpos, shape.theta, True))
        dOt = orc.bf16_round((dout[tpos].to(torch.float64).numpy() @ Wo).reshape(T, H, D_HEAD))
        dq = np.empty((T, H, D_HEAD))
        dk = np.zeros((T, Hkv, D_HEAD))
        dv = np.zeros((T, Hkv, D_HEAD))
        for h in range(H):
            kh, vh = K[:, h // g], V[:, h // g]
            o_t, l_t = orc.attention_head_rows(Qt[:, h], tpos, kh, vh, scale)
            o_t = orc.bf16_round(o_t)
            dq[:, h] = orc.attention_dq_rows(Qt[:, h], tpos, kh, vh, dOt[:, h], o_t, l_t, scale)
            a, b = orc.attention_dkv_tail(Qt[:, h], kh[tpos], vh[tpos], dOt[:, h], o_t, l_t, scale)
            dk[:, h // g] += a
            dv[:, h // g] += b
        dq = orc.rope_apply(dq, tpos, shape.theta, inverse=True)
        dk = orc.rope_apply(dk, tpos, shape.theta, inverse=True)
        dqkv = np.concatenate([dq.reshape(T, -1), dk.reshape(T, -1), dv.reshape(T, -1)], 1)
        assert_close(f64(dx[tpos]), dqkv @ w.to(torch.float64).numpy(), "dx tail rows")

    if dwo_head is not None:
        h = dwo_head
        allpos = np.arange(L)
        Qh = np.empty((L, D_HEAD))
        for s0 in range(0, L, 16384):
            pos = allpos[s0:s0 + 16384]
            Qh[pos] = _proj_rows(x, w, np.arange(h * D_HEAD, (h + 1) * D_HEAD), pos, shape.theta, True)[:, 0]
        Oh, _ = orc.attention_head_rows(orc.bf16_round(Qh), allpos, K[:, h // g], V[:, h // g], scale)
        Oh = orc.bf16_round(Oh)
        ref = dout.to(torch.float64).numpy().T @ Oh
        assert_close(f64(dwo[:, h * D_HEAD:(h + 1) * D_HEAD]), ref, "dWo head columns", weight_grad=True)


def _assert_bit_exact(a, b, what):
    for x, y, n in zip(a, b, ("out", "lse", "dx", "dWqkv", "dWo")):
        assert torch.equal(x, y), f"{what}: {n} differs"


def test_llama3_8b_layer_L32768():
    """D=4096, H=32, Hkv=8, U=8 (the benchmark workload), and U=32 bit-exact."""
    shape = synth.LLAMA8B
    inputs = synth.layer_inputs(shape)
    res = _run_layer(shape, 8, inputs)
    _check_layer_rows(shape, inputs, res, _rows(shape.L), tail=256, dwo_head=5)
    _assert_bit_exact(res, _run_layer(shape, 32, inputs), "U=8 vs U=32")


def test_qwen32b_shape_layer_L131072_u_sweep():
    """D=5120, H=64, Hkv=8, U in {64, 16, 8}: identical bits, oracle rows."""
    shape = synth.LayerShape(L=131072, D=5120, H=64, Hkv=8, U=8)
    inputs = synth.layer_inputs(shape)
    res8 = _run_layer(shape, 8, inputs)
    _check_layer_rows(shape, inputs, res8, _rows(shape.L, n=6), tail=128)
    for U in (16, 64):
        _assert_bit_exact(res8, _run_layer(shape, U, inputs), f"U=8 vs U={U}")


@pytest.mark.parametrize("L", [65536, 262144])
def test_long_context_sweep_layer(L):
    """Llama-3-8B shape, U=4 (U < g): oracle rows and tail, U=8 bit-exact."""
    shape = synth.LayerShape(L=L, D=4096, H=32, Hkv=8, U=4)
    inputs = synth.layer_inputs(shape)
    res = _run_layer(shape, 4, inputs)
    _check_layer_rows(shape, inputs, res, _rows(L, n=6), tail=128)
    _assert_bit_exact(res, _run_layer(shape, 8, inputs), "U=4 vs U=8")


def test_long_context_sweep_layer_L1M_early_rows():
    """L = 1,048,576, U=4: the full-size run; oracle rows in the first 32K
    positions (a row needs every earlier K/V), finite outputs everywhere."""
    shape = synth.LayerShape(L=1 << 20, D=4096, H=32, Hkv=8, U=4)
    inputs = synth.layer_inputs(shape)
    res = _run_layer(shape, 4, inputs)
    for t in res:
        assert torch.isfinite(t.float()).all()
    rng = np.random.default_rng(1)
    uni = np.unique(rng.integers(0, 32768, 12)).astype(np.int64)
    edge = np.array([0, 1, 127, 128, 4095, 4096, 32767], dtype=np.int64)
    _check_layer_rows(shape, inputs, res, (uni, edge), tail=0)


def test_ulysses_slice_core_L1M():
    """Core entry, L = 1,048,576, H=4, Hkv=1, U=1 (U < g: carried dK/dV):
    oracle rows of O/LSE/dQ, dK/dV of the last 512 keys, U=4 bit-exact."""
    L, H, Hkv = 1 << 20, 4, 1
    q, k, v, do = synth.core_inputs(L, H, Hkv)
    qd, kd, vd, dod = (t.to("cuda:0") for t in (q, k, v, do))
    outs = {}
    for U in (1, 4):
        cfg = upipe.Config(L=L, H=H, Hkv=Hkv, U=U)
        o, lse = upipe.core_forward(cfg, qd, kd, vd)
        dq, dk, dv = upipe.core_backward(cfg, qd, kd, vd, o, lse, dod)
        torch.cuda.synchronize()
        status_ok()
        outs[U] = tuple(t.cpu() for t in (o, lse, dq, dk, dv))
        del o, lse, dq, dk, dv
    for a, b, n in zip(outs[1], outs[4], ("o", "lse", "dq", "dk", "dv")):
        assert torch.equal(a, b), f"U=1 vs U=4: {n} differs"
    o, lse, dq, dk, dv = outs[1]
    scale = 1 / math.sqrt(D_HEAD)
    K = k[:, 0].to(torch.float64).numpy()
    V = v[:, 0].to(torch.float64).numpy()
    uni, edge = _rows(L, n=24)
    T = 512
    tpos = np.arange(L - T, L)
    dk_t = np.zeros((T, D_HEAD))
    dv_t = np.zeros((T, D_HEAD))
    for rows, kind in ((uni, "uniform"), (edge, "edge")):
        ro = np.empty((len(rows), H, D_HEAD))
        rl = np.empty((H, len(rows)))
        rdq = np.empty((len(rows), H, D_HEAD))
        for h in range(H):
            qr = q[rows, h].to(torch.float64).numpy()
            ro[:, h], rl[h] = orc.attention_head_rows(qr, rows, K, V, scale)
            ob = orc.bf16_round(ro[:, h])  # o enters the backward as a bf16 tensor
            dor = do[rows, h].to(torch.float64).numpy()
            rdq[:, h] = orc.attention_dq_rows(qr, rows, K, V, dor, ob, rl[h], scale)
        check = assert_close if kind == "uniform" else assert_max_abs
        check(f64(o[rows]), ro, f"o {kind} rows")
        check(f64(lse[:, rows]), rl, f"lse {kind} rows")
        check(f64(dq[rows]), rdq, f"dq {kind} rows")
    for h in range(H):
        qt = q[tpos, h].to(torch.float64).numpy()
        ot, lt = orc.attention_head_rows(qt, tpos, K, V, scale)
        ot = orc.bf16_round(ot)
        a, b = orc.attention_dkv_tail(qt, K[tpos], V[tpos], do[tpos, h].to(torch.float64).numpy(), ot, lt, scale)
        dk_t += a
        dv_t += b
    assert_close(f64(dk[tpos, 0]), dk_t, "dk tail")
    assert_close(f64(dv[tpos, 0]), dv_t, "dv tail")
