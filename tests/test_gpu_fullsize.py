"""GPU parity at the full workload sizes, on outputs the fp64 oracle can
compute one by one, plus bit-exactness of every chunk size U at those sizes.

Sampled checks (oracle fp64 in its precision-model mode -- every contraction
input rounded to bf16 -- unless a check says "plain"; the GPU run is the
full-size run):
 * forward rows: out and LSE of sampled query positions drawn uniformly
   over the whole sequence (each needs that row's Q and the K/V of every
   earlier position), plus edge rows (first, tile boundaries, last);
 * backward tail: under the causal mask the last T keys are seen only by the
   last T queries, so dQ, dK, dV -- and hence dx -- of the last T positions
   follow from those T rows alone (plus their O/LSE rows);
 * one head's columns of dWo (needs that head's O for every row);
 * one KV group's rows of dWqkv (its query heads, its K and V rows: needs
   the group's whole attention backward, O(L^2 d) per head).
Everything else at these sizes is pinned by bit-exactness against another
chunk size and by the small-size full parity tests.
"""

import math
import os
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from oracle import upipe_oracle as orc
from tests.gpu_common import ensure_lib, f64, status_ok
from tests.tolerance import assert_close, assert_close_plain, assert_max_abs

pytestmark = pytest.mark.gpu

D_HEAD = 128
NAMES = ("out", "lse", "dx", "dWqkv", "dWo")


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


def _kv_all(x, W, shape, upto, block=16384, exact=True):
    """fp64 K (RoPE'd) and V [upto, Hkv, d] from x[:upto], blockwise: the
    exact values (or None) and their bf16 roundings (the precision model's
    stored K and V), each block rounded as it is computed."""
    H, Hkv = shape.H, shape.Hkv
    rk = np.arange(H * D_HEAD, (H + Hkv) * D_HEAD)
    rv = np.arange((H + Hkv) * D_HEAD, (H + 2 * Hkv) * D_HEAD)
    K = np.empty((upto, Hkv, D_HEAD)) if exact else None
    V = np.empty((upto, Hkv, D_HEAD)) if exact else None
    Kb = np.empty((upto, Hkv, D_HEAD))
    Vb = np.empty((upto, Hkv, D_HEAD))
    for s0 in range(0, upto, block):
        pos = np.arange(s0, min(upto, s0 + block))
        k = _proj_rows(x, W, rk, pos, shape.theta, True)
        v = _proj_rows(x, W, rv, pos, shape.theta, False)
        Kb[pos], Vb[pos] = orc.bf16_round(k), orc.bf16_round(v)
        if exact:
            K[pos], V[pos] = k, v
    return K, V, Kb, Vb


def _nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


def _run_layer(shape, U, inputs, on_device=None, peaks=None, keep_o=False):
    """Full-size forward + backward.  Returns the five results on the host,
    or on the device when `on_device` (then the device inputs too).  With a
    dict `peaks`, records the device high-water mark of each pass's
    intermediate memory (the helpers size and allocate the workspace; the
    caller-visible outputs are subtracted)."""
    cfg = upipe.Config(L=shape.L, D=shape.D, H=shape.H, Hkv=shape.Hkv, U=U, rope_theta=shape.theta)
    dev_in = on_device if on_device is not None else tuple(t.to("cuda:0") for t in inputs)
    xd, wd, wod, dd = dev_in
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    out, lse, kept = upipe.layer_forward(cfg, xd, wd, wod, keep_o=keep_o)
    torch.cuda.synchronize()
    fwd_peak = torch.cuda.max_memory_allocated() - base - _nbytes(out, lse)
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    dx, dwqkv, dwo = upipe.layer_backward(cfg, xd, wd, wod, dd, lse, kept)
    torch.cuda.synchronize()
    bwd_peak = torch.cuda.max_memory_allocated() - base - _nbytes(dx, dwqkv, dwo)
    status_ok()
    if peaks is not None:
        peaks[U] = (fwd_peak, bwd_peak)
    res = (out, lse, dx, dwqkv, dwo)
    if on_device is not None:
        return res
    res = tuple(t.cpu() for t in res)
    del xd, wd, wod, dd, dev_in, out, lse, dx, dwqkv, dwo
    torch.cuda.empty_cache()
    return res


def _fwd_rows(Q, K, V, rows, g, scale):
    """Forward output rows (the forward's own P V keeps P exact)."""
    H = Q.shape[1]
    O = np.empty((len(rows), H, D_HEAD))
    Lr = np.empty((H, len(rows)))
    for h in range(H):
        O[:, h], Lr[h] = orc.attention_head_rows(Q[:, h], rows, K[:, h // g], V[:, h // g], scale)
    return O, Lr


def _tail(Qt, dOt, K, V, tpos, g, scale, bf, theta, kept_o=False):
    """dQ, dK, dV of the last T positions (RoPE undone on dQ, dK).  Heads are
    independent, so they run on a thread pool (NumPy releases the GIL in its
    matrix products and element-wise loops); each head's dK/dV share is
    summed into its KV head afterwards, in head order.  kept_o: the backward
    reads the forward's own O (P exact in P V) instead of O recomputed from
    the LSE."""
    T, H = Qt.shape[0], Qt.shape[1]
    Hkv = K.shape[1]
    rnd = orc.bf16_round if bf else (lambda a: a)
    dq = np.empty((T, H, D_HEAD))
    dk = np.zeros((T, Hkv, D_HEAD))
    dv = np.zeros((T, Hkv, D_HEAD))

    def head(h):
        kh, vh = K[:, h // g], V[:, h // g]
        # O recomputed from the LSE, as the backward does (or the kept one)
        o_t, l_t = orc.attention_head_rows(Qt[:, h], tpos, kh, vh, scale, p_bf16=bf and not kept_o)
        o_t = rnd(o_t)
        dq_h = orc.attention_dq_rows(Qt[:, h], tpos, kh, vh, dOt[:, h], o_t, l_t, scale, bf16_operands=bf)
        a, b = orc.attention_dkv_tail(Qt[:, h], kh[tpos], vh[tpos], dOt[:, h], o_t, l_t, scale, bf16_operands=bf)
        return dq_h, a, b

    with ThreadPoolExecutor(max_workers=min(H, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(head, range(H)))
    for h, (dq_h, a, b) in enumerate(parts):
        dq[:, h] = dq_h
        dk[:, h // g] += a
        dv[:, h // g] += b
    dq = orc.rope_apply(dq, tpos, theta, inverse=True)
    dk = orc.rope_apply(dk, tpos, theta, inverse=True)
    return np.concatenate([dq.reshape(T, -1), dk.reshape(T, -1), dv.reshape(T, -1)], 1)


def _check_layer_rows(shape, inputs, res, fwd_rows, tail, dwo_head=None, plain=False, kept_o=False, kv=None):
    """Sampled forward rows, the backward tail and one head's dWo columns
    against the precision-model oracle (and, with `plain`, against the plain
    fp64 definition as well).  kept_o: the backward read the forward's own
    O (O kept in host memory).  kv: (K, V, Kb, Vb) of an earlier call on the
    same inputs."""
    x, w, wo, dout = inputs
    out, lse, dx, dwqkv, dwo = res
    H, Hkv, L = shape.H, shape.Hkv, shape.L
    g = H // Hkv
    scale = 1 / math.sqrt(D_HEAD)
    wq_rows = np.arange(H * D_HEAD)
    uni, edge = fwd_rows
    fwd_rows = np.unique(np.concatenate([uni, edge]))
    need = L if (tail or dwo_head is not None) else int(fwd_rows.max()) + 1
    K, V, Kb, Vb = kv if kv is not None else _kv_all(x, w, shape, need, exact=plain)
    Wo = wo.to(torch.float64).numpy()
    W = w.to(torch.float64).numpy()
    iu = np.searchsorted(fwd_rows, uni)
    ie = np.searchsorted(fwd_rows, edge)

    # forward rows
    Q = _proj_rows(x, w, wq_rows, fwd_rows, shape.theta, True)
    Or, Lr = _fwd_rows(orc.bf16_round(Q), Kb, Vb, fwd_rows, g, scale)
    ref_out = orc.bf16_round(Or).reshape(len(fwd_rows), -1) @ Wo.T
    got_out, got_lse = f64(out[uni]), f64(lse[:, uni])
    assert_close(got_out, ref_out[iu], "out rows")
    assert_close(got_lse, Lr[:, iu], "lse rows")
    assert_max_abs(f64(out[edge]), ref_out[ie], "out edge rows")
    assert_max_abs(f64(lse[:, edge]), Lr[:, ie], "lse edge rows")
    if plain:
        Op, Lp = _fwd_rows(Q, K, V, fwd_rows, g, scale)
        plain_out = Op.reshape(len(fwd_rows), -1) @ Wo.T
        assert_close_plain(got_out, plain_out[iu], ref_out[iu], "out rows")
        assert_close_plain(got_lse, Lp[:, iu], Lr[:, iu], "lse rows")

    if tail:
        T = tail
        tpos = np.arange(L - T, L)
        Qt = _proj_rows(x, w, wq_rows, tpos, shape.theta, True)
        dOt = (dout[tpos].to(torch.float64).numpy() @ Wo).reshape(T, H, D_HEAD)
        dqkv = _tail(orc.bf16_round(Qt), orc.bf16_round(dOt), Kb, Vb, tpos, g, scale, True, shape.theta, kept_o)
        got = f64(dx[tpos])
        assert_close(got, dqkv @ W, "dx tail rows")
        if plain:
            dqkv_p = _tail(Qt, dOt, K, V, tpos, g, scale, False, shape.theta)
            assert_close_plain(got, dqkv_p @ W, dqkv @ W, "dx tail rows")

    if dwo_head is not None:
        h = dwo_head
        allpos = np.arange(L)
        Qh = np.empty((L, D_HEAD))
        for s0 in range(0, L, 16384):
            pos = allpos[s0:s0 + 16384]
            Qh[pos] = _proj_rows(x, w, np.arange(h * D_HEAD, (h + 1) * D_HEAD), pos, shape.theta, True)[:, 0]
        Oh, _ = orc.attention_head_rows(orc.bf16_round(Qh), allpos, Kb[:, h // g], Vb[:, h // g], scale,
                                        p_bf16=not kept_o)  # the backward's O: recomputed from the LSE, or kept
        ref = dout.to(torch.float64).numpy().T @ orc.bf16_round(Oh)
        assert_close(f64(dwo[:, h * D_HEAD:(h + 1) * D_HEAD]), ref, "dWo head columns", weight_grad=True)
    return K, V, Kb, Vb


def _check_dwqkv_group(shape, inputs, dwqkv, kv, Kb, Vb):
    """dWqkv rows of KV group `kv` -- its g query heads' rows, its K rows and
    its V rows -- from the group's whole attention backward (oracle in its
    precision-model mode; Kb, Vb are the stored bf16 K and V)."""
    x, w, wo, dout = inputs
    H, Hkv, L = shape.H, shape.Hkv, shape.L
    g = H // Hkv
    heads = np.arange(kv * g, (kv + 1) * g)
    allpos = np.arange(L)
    q_rows = np.concatenate([np.arange(h * D_HEAD, (h + 1) * D_HEAD) for h in heads])
    Q = np.empty((L, g, D_HEAD))
    for s0 in range(0, L, 16384):
        pos = allpos[s0:s0 + 16384]
        Q[pos] = _proj_rows(x, w, q_rows, pos, shape.theta, True)
    Q = orc.bf16_round(Q)
    Kj, Vj = Kb[:, kv:kv + 1], Vb[:, kv:kv + 1]
    O, lse = orc.attention_core_fwd(Q, Kj, Vj, p_bf16=True)  # the backward's O, from the LSE
    O = orc.bf16_round(O)
    Wo = wo.to(torch.float64).numpy()
    cols = np.concatenate([np.arange(h * D_HEAD, (h + 1) * D_HEAD) for h in heads])
    dO = orc.bf16_round((dout.to(torch.float64).numpy() @ Wo[:, cols]).reshape(L, g, D_HEAD))
    dq, dk, dv = orc.attention_core_bwd(Q, Kj, Vj, O, lse, dO, bf16_operands=True)
    dq = orc.rope_apply(dq, allpos, shape.theta, inverse=True)
    dk = orc.rope_apply(dk, allpos, shape.theta, inverse=True)
    X = x.to(torch.float64).numpy()
    ref_q = dq.reshape(L, -1).T @ X
    ref_k = dk.reshape(L, -1).T @ X
    ref_v = dv.reshape(L, -1).T @ X
    got = f64(dwqkv)
    assert_close(got[q_rows], ref_q, f"dWqkv rows of q heads {heads[0]}..{heads[-1]}", weight_grad=True)
    rk = slice((H + kv) * D_HEAD, (H + kv + 1) * D_HEAD)
    rv = slice((H + Hkv + kv) * D_HEAD, (H + Hkv + kv + 1) * D_HEAD)
    assert_close(got[rk], ref_k, f"dWqkv rows of k head {kv}", weight_grad=True)
    assert_close(got[rv], ref_v, f"dWqkv rows of v head {kv}", weight_grad=True)


def _assert_bit_exact(a, b, what):
    for x, y, n in zip(a, b, NAMES):
        assert torch.equal(x, y), f"{what}: {n} differs"


def test_llama3_8b_layer_L32768():
    """D=4096, H=32, Hkv=8, U=8 (Llama-3-8B layer shape): oracle rows, tail,
    dWo columns and one KV group's dWqkv rows, plain-definition figures;
    U=32 bit-exact; O kept in host memory checked against its own model."""
    shape = synth.LLAMA8B
    inputs = synth.layer_inputs(shape)
    res = _run_layer(shape, 8, inputs)
    kv = _check_layer_rows(shape, inputs, res, _rows(shape.L), tail=256, dwo_head=5, plain=True)
    _check_dwqkv_group(shape, inputs, res[3], 1, kv[2], kv[3])
    _assert_bit_exact(res, _run_layer(shape, 32, inputs), "U=8 vs U=32")
    # O kept in page-locked host memory: the forward's bits, and the backward
    # (dx tail, one head's dWo columns) against the kept-O model
    res_h = _run_layer(shape, 8, inputs, keep_o="host")
    assert torch.equal(res_h[0], res[0]) and torch.equal(res_h[1], res[1])
    _check_layer_rows(shape, inputs, res_h, _rows(shape.L, n=4), tail=128, dwo_head=21, kept_o=True, kv=kv)


def test_qwen32b_shape_layer_L131072_u_sweep():
    """D=5120, H=64, Hkv=8, U in {64, 16, 8}: identical bits, oracle rows,
    and the measured intermediate memory of each U against the library's
    arithmetic: chunk bytes scale as U/H, so U=8 keeps 12.5% of the
    unchunked chunk buffers (the abstract's 87.5% reduction for 32B
    models)."""
    shape = synth.LayerShape(L=131072, D=5120, H=64, Hkv=8, U=8)
    inputs = synth.layer_inputs(shape)
    peaks = {}
    res8 = _run_layer(shape, 8, inputs, peaks=peaks)
    kv = _check_layer_rows(shape, inputs, res8, _rows(shape.L, n=6), tail=128)
    # O kept in page-locked host memory (the benchmark's mode): eight chunks
    # through the two staging buffers; the forward is the recomputing
    # forward's bit for bit, the backward is checked against the kept-O model.
    res_h = _run_layer(shape, 8, inputs, keep_o="host")
    assert torch.equal(res_h[0], res8[0]) and torch.equal(res_h[1], res8[1])
    _check_layer_rows(shape, inputs, res_h, _rows(shape.L, n=6), tail=128, kept_o=True, kv=kv)
    _assert_bit_exact(res_h, _run_layer(shape, 16, inputs, keep_o="host"), "O in host memory, U=8 vs U=16")
    for U in (16, 64):
        _assert_bit_exact(res8, _run_layer(shape, U, inputs, peaks=peaks), f"U=8 vs U={U}")
    chunk = {}
    for U, (fwd, bwd) in sorted(peaks.items()):
        cfg = upipe.Config(L=shape.L, D=shape.D, H=shape.H, Hkv=shape.Hkv, U=U)
        ws_f, ws_b = upipe.workspace_bytes(cfg, 0), upipe.workspace_bytes(cfg, 1)
        cb, fb = upipe.activation_bytes(cfg, 1)
        chunk[U] = cb
        print(f"[memory] U={U}: measured fwd {fwd} B (library {ws_f}), bwd {bwd} B (library {ws_b}); "
              f"bwd chunk {cb} B + fixed {fb} B")
        # the device high-water mark is the library's workspace (torch's
        # allocator rounds a large block up to a multiple of 2 MiB)
        assert ws_f <= fwd <= ws_f + (2 << 20)
        assert ws_b <= bwd <= ws_b + (2 << 20)
    for U in (8, 16):
        assert chunk[U] * 64 == chunk[64] * U
    print(f"[memory] U=8 chunk buffers: {chunk[8] / chunk[64]:.3f} of U=64 "
          f"({1 - chunk[8] / chunk[64]:.1%} less)")
    assert 1 - chunk[8] / chunk[64] == pytest.approx(0.875, abs=0)


@pytest.mark.parametrize("L", [65536, 262144])
def test_long_context_sweep_layer(L):
    """Llama-3-8B shape, U=4 (U < g): oracle rows and tail, U=8 bit-exact."""
    shape = synth.LayerShape(L=L, D=4096, H=32, Hkv=8, U=4)
    inputs = synth.layer_inputs(shape)
    res = _run_layer(shape, 4, inputs)
    _check_layer_rows(shape, inputs, res, _rows(L, n=6), tail=128)
    _assert_bit_exact(res, _run_layer(shape, 8, inputs), "U=4 vs U=8")


def _gather(res, rows, tail):
    """The sampled rows of a device run, on the host: out rows, LSE columns,
    the dx tail (the sampled checks need nothing else)."""
    out, lse, dx, dwqkv, dwo = res
    r = torch.as_tensor(rows, device=out.device)
    t = torch.arange(out.shape[0] - tail, out.shape[0], device=out.device)
    return out[r].cpu(), lse[:, r].cpu(), dx[t].cpu()


def test_long_context_sweep_layer_L1M_and_L2M(monkeypatch):
    """Llama-3-8B shape, U=4 (U < g), at L = 1,048,576 and L = 2,097,152 (the
    long-context sweep's largest length; the unchunked U=32 run does not fit
    at 2M: its workspace alone is ~128 GiB on top of ~96 GiB of layer
    tensors and fp32 carry).  At each length: the U=4 and U=8 runs compared
    bit for bit on the device, every output finite, oracle rows drawn
    uniformly over the whole sequence plus edge rows, and the last-128 tail
    of dx.  The 1M inputs are the first 1M rows of the 2M inputs, so the
    fp64 K/V projection is computed once.  The inputs are drawn on the
    device (seeded CUDA generator) and copied to the host for the oracle:
    both sides see the same bf16 values."""
    t_start = time.time()
    big = synth.LayerShape(L=1 << 21, D=4096, H=32, Hkv=8, U=4)
    xd_all, wd, wod, dd_all = synth.layer_inputs(big, device="cuda:0")
    x, w, wo, dout = (t.cpu() for t in (xd_all, wd, wod, dd_all))
    # Sampled rows in blocks of 32 per head (the streamed blocking changes no
    # result: see the oracle pins), so that the heads running in parallel
    # in _tail each hold a few 32 x L score blocks.
    monkeypatch.setattr(orc, "ROW_BLOCK", 32)
    # The fp64 K/V projection of all 2M rows (CPU) runs on a second thread
    # while the GPU runs below: BLAS and CUDA waits both release the GIL.
    kv = {}
    worker = threading.Thread(target=lambda: kv.update(r=_kv_all(x, w, big, big.L, exact=False)))
    worker.start()
    H, Hkv, g = big.H, big.Hkv, big.H // big.Hkv
    scale = 1 / math.sqrt(D_HEAD)
    Wo = wo.to(torch.float64).numpy()
    W = w.to(torch.float64).numpy()
    wq_rows = np.arange(H * D_HEAD)
    T = 128
    sampled = {}
    for L in (1 << 20, 1 << 21):
        shape = synth.LayerShape(L=L, D=4096, H=32, Hkv=8, U=4)
        dev_in = (xd_all[:L], wd, wod, dd_all[:L])
        res4 = _run_layer(shape, 4, None, on_device=dev_in)
        res8 = _run_layer(shape, 8, None, on_device=dev_in)
        _assert_bit_exact(res4, res8, f"L={L}: U=4 vs U=8")
        del res8
        for t, n in zip(res4, NAMES):
            assert bool(torch.isfinite(t).all()), f"L={L}: non-finite {n}"
        uni, edge = _rows(L, n=8, seed=L)
        rows = np.unique(np.concatenate([uni, edge]))
        sampled[L] = (uni, edge, rows, *_gather(res4, rows, T))
        del res4
        torch.cuda.empty_cache()
        print(f"[time] L={L}: GPU runs done at {time.time() - t_start:.0f} s")
    del xd_all, dd_all, dev_in
    torch.cuda.empty_cache()
    worker.join()
    _, _, Kb, Vb = kv["r"]
    print(f"[time] K/V projection joined at {time.time() - t_start:.0f} s")
    for L in (1 << 20, 1 << 21):
        uni, edge, rows, out_r, lse_r, dx_t = sampled[L]
        # forward rows
        Q = orc.bf16_round(_proj_rows(x, w, wq_rows, rows, big.theta, True))
        Or, Lr = _fwd_rows(Q, Kb[:L], Vb[:L], rows, g, scale)
        ref_out = orc.bf16_round(Or).reshape(len(rows), -1) @ Wo.T
        iu, ie = np.searchsorted(rows, uni), np.searchsorted(rows, edge)
        assert_close(f64(out_r[iu]), ref_out[iu], f"L={L}: out rows")
        assert_close(f64(lse_r[:, iu]), Lr[:, iu], f"L={L}: lse rows")
        assert_max_abs(f64(out_r[ie]), ref_out[ie], f"L={L}: out edge rows")
        assert_max_abs(f64(lse_r[:, ie]), Lr[:, ie], f"L={L}: lse edge rows")
        # backward tail
        tpos = np.arange(L - T, L)
        Qt = orc.bf16_round(_proj_rows(x, w, wq_rows, tpos, big.theta, True))
        dOt = orc.bf16_round((dout[tpos].to(torch.float64).numpy() @ Wo).reshape(T, H, D_HEAD))
        dqkv = _tail(Qt, dOt, Kb[:L], Vb[:L], tpos, g, scale, True, big.theta)
        assert_close(f64(dx_t), dqkv @ W, f"L={L}: dx tail rows")
        print(f"[time] L={L}: oracle checks done at {time.time() - t_start:.0f} s")


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
            # the core forward's output (P exact); o enters the backward as a bf16 tensor
            ro[:, h], rl[h] = orc.attention_head_rows(qr, rows, K, V, scale)
            ob = orc.bf16_round(ro[:, h])
            dor = do[rows, h].to(torch.float64).numpy()
            rdq[:, h] = orc.attention_dq_rows(qr, rows, K, V, dor, ob, rl[h], scale, bf16_operands=True)
        check = assert_close if kind == "uniform" else assert_max_abs
        check(f64(o[rows]), ro, f"o {kind} rows")
        check(f64(lse[:, rows]), rl, f"lse {kind} rows")
        check(f64(dq[rows]), rdq, f"dq {kind} rows")
    for h in range(H):
        qt = q[tpos, h].to(torch.float64).numpy()
        ot, lt = orc.attention_head_rows(qt, tpos, K, V, scale)
        ot = orc.bf16_round(ot)
        a, b = orc.attention_dkv_tail(qt, K[tpos], V[tpos], do[tpos, h].to(torch.float64).numpy(), ot, lt, scale,
                                      bf16_operands=True)
        dk_t += a
        dv_t += b
    assert_close(f64(dk[tpos, 0]), dk_t, "dk tail")
    assert_close(f64(dv[tpos, 0]), dv_t, "dv tail")

