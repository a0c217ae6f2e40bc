"""GPU parity of the sequence-tiled SwiGLU MLP and LM-head cross-entropy
(include/upipe.h: upipe_mlp_fwd / _bwd, upipe_ce_fwd_bwd) against the fp64
oracle (oracle/alst_oracle.py), through the C ABI: element by element at
sizes spanning several tiles with ragged tails, against the precision-model
oracle (bf16 intermediates) and the plain fp64 definition; identical bits
for every tile size; and at the Llama-3-8B MLP and vocabulary sizes, sampled
rows and weight-gradient columns the oracle computes one by one."""

import numpy as np
import pytest
import torch

from headwise_chunked_context_gb300 import synth, upipe
from oracle import alst_oracle as alst
from tests.gpu_common import ensure_lib, f64, status_ok
from tests.tolerance import assert_close, assert_close_plain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _mlp(L, D, F, T, inputs=None):
    x, wgu, wd, dy = inputs if inputs is not None else synth.mlp_inputs(L, D, F)
    xd, wgud, wdd, dyd = (t.to("cuda:0") for t in (x, wgu, wd, dy))
    y = upipe.mlp_forward(xd, wgud, wdd, T)
    dx, dwgu, dwd = upipe.mlp_backward(xd, wgud, wdd, dyd, T)
    torch.cuda.synchronize()
    status_ok()
    return (x, wgu, wd, dy), (y, dx, dwgu, dwd)


@pytest.mark.parametrize("L,D,F,T", [(300, 256, 384, 128), (1024, 512, 1024, 256), (129, 128, 256, 128),
                                     (1, 128, 128, 128), (640, 256, 256, 512)])
def test_mlp_matches_oracle(L, D, F, T):
    (x, wgu, wd, dy), outs = _mlp(L, D, F, T)
    x, wgu, wd, dy = (f64(t) for t in (x, wgu, wd, dy))
    got = [f64(t) for t in outs]
    my, _ = alst.mlp_fwd(x, wgu, wd, bf16_operands=True)
    model = (my, *alst.mlp_bwd(x, wgu, wd, dy, bf16_operands=True))
    py, _ = alst.mlp_fwd(x, wgu, wd)
    plain = (py, *alst.mlp_bwd(x, wgu, wd, dy))
    for g_, m, p, n, wg in zip(got, model, plain, ("y", "dx", "dWgu", "dWd"), (False, False, True, True)):
        assert_close(g_, m, f"mlp {n}", weight_grad=wg)
        assert_close_plain(g_, p, m, f"mlp {n}", weight_grad=wg)


def test_mlp_every_tile_size_gives_identical_bits():
    L, D, F = 1000, 256, 512
    inputs = synth.mlp_inputs(L, D, F)
    _, ref = _mlp(L, D, F, 1024, inputs)
    for T in (128, 256, 384, 512):
        _, outs = _mlp(L, D, F, T, inputs)
        for a, b, n in zip(ref, outs, ("y", "dx", "dWgu", "dWd")):
            assert torch.equal(a, b), f"T={T}: {n} differs from the single-tile run"


def _ce(L, D, V, T, inputs=None, scale=None):
    h, w, labels = inputs if inputs is not None else synth.ce_inputs(L, D, V)
    if scale is None:
        scale = 1.0 / max(1, int((labels >= 0).sum()))
    hd, wdev, ld = (t.to("cuda:0") for t in (h, w, labels))
    loss, dh, dw = upipe.ce_loss(hd, wdev, ld, scale, T)
    torch.cuda.synchronize()
    status_ok()
    return (h, w, labels, scale), (loss, dh, dw)


@pytest.mark.parametrize("L,D,V,T", [(300, 256, 1024, 128), (77, 128, 512, 128), (513, 256, 2048, 256),
                                     (1, 128, 128, 128)])
def test_ce_matches_oracle(L, D, V, T):
    (h, w, labels, scale), outs = _ce(L, D, V, T)
    h, w = f64(h), f64(w)
    lab = labels.numpy()
    got = [f64(t) for t in outs]
    model = alst.ce_fwd_bwd(h, w, lab, scale, bf16_operands=True)
    plain = alst.ce_fwd_bwd(h, w, lab, scale)
    for g_, m, p, n, wg in zip(got, model, plain, ("loss", "dh", "dW"), (False, False, True)):
        assert_close(g_, m, f"ce {n}", weight_grad=wg)
        assert_close_plain(g_, p, m, f"ce {n}", weight_grad=wg)
    assert np.all(got[0][lab < 0] == 0) and np.all(got[1][lab < 0] == 0)


def test_ce_every_tile_size_gives_identical_bits_and_bad_labels_are_loud():
    L, D, V = 700, 256, 1024
    h, w, labels = synth.ce_inputs(L, D, V)
    labels[5] = V  # outside the vocabulary: NaN loss, no gradient
    inputs = (h, w, labels)
    _, ref = _ce(L, D, V, 768, inputs, scale=0.01)
    assert torch.isnan(ref[0][5]) and torch.all(ref[1][5] == 0)
    assert torch.isfinite(ref[0][labels != V]).all()
    for T in (128, 256, 384):
        _, outs = _ce(L, D, V, T, inputs, scale=0.01)
        assert torch.equal(ref[0].nan_to_num(), outs[0].nan_to_num()), f"T={T}: loss differs"
        for a, b, n in zip(ref[1:], outs[1:], ("dh", "dW")):
            assert torch.equal(a, b), f"T={T}: {n} differs from the single-tile run"


# ------------------------------------------------------------- full size

def _rows(L, n, seed):
    r = np.random.default_rng(seed)
    return np.unique(np.concatenate([r.integers(0, L, n), [0, L - 1]]))


@pytest.mark.parametrize("L,D,F,T", [(32768, 4096, 14336, 8192), (65536, 5120, 27648, 16384)])
def test_full_size_mlp_sampled_rows_and_columns(L, D, F, T):
    """The Llama-3-8B MLP (D=4096, F=14336) and the 32B family's (D=5120,
    F=27648) in tiles of T rows: y and dx rows, dWd columns and dWgu rows
    against the precision-model oracle, computed one by one; one tile of all
    L rows gives identical bits."""
    x, wgu, wd, dy = synth.mlp_inputs(L, D, F, device="cuda:0")
    y = upipe.mlp_forward(x, wgu, wd, T)
    dx, dwgu, dwd = upipe.mlp_backward(x, wgu, wd, dy, T)
    torch.cuda.synchronize()
    status_ok()
    X, WGU, WD, DY = (t.to("cpu", torch.float64).numpy() for t in (x, wgu, wd, dy))
    rows = _rows(L, 10, 0)
    my, _ = alst.mlp_fwd(X[rows], WGU, WD, bf16_operands=True)
    mdx, _, _ = alst.mlp_bwd(X[rows], WGU, WD, DY[rows], bf16_operands=True, weight_grads=False)
    assert_close(f64(y[rows]), my, "mlp y rows")
    assert_close(f64(dx[rows]), mdx, "mlp dx rows")
    # dWd[:, f] = dy^T H[:, f] and dWgu[f] = dG[:, f]^T x (gate row), dWgu[F + f] = dU[:, f]^T x
    cols = np.array([0, 777, F - 1])
    g = X @ WGU[cols].T
    u = X @ WGU[F + cols].T
    s = 1.0 / (1.0 + np.exp(-g))
    h = alst.bf16_round(g * s * u)
    dh = alst.bf16_round(DY @ WD[:, cols])
    dg = alst.bf16_round(dh * u * s * (1.0 + g * (1.0 - s)))
    du = alst.bf16_round(dh * g * s)
    assert_close(f64(dwd[:, cols]), DY.T @ h, "mlp dWd columns", weight_grad=True)
    assert_close(f64(dwgu[cols]), dg.T @ X, "mlp dWgu gate rows", weight_grad=True)
    assert_close(f64(dwgu[F + cols]), du.T @ X, "mlp dWgu up rows", weight_grad=True)
    y1 = upipe.mlp_forward(x, wgu, wd, L)
    dx1, dwgu1, dwd1 = upipe.mlp_backward(x, wgu, wd, dy, L)
    for a, b, n in zip((y, dx, dwgu, dwd), (y1, dx1, dwgu1, dwd1), ("y", "dx", "dWgu", "dWd")):
        assert torch.equal(a, b), f"T={T} vs one tile: {n} differs"


@pytest.mark.parametrize("L,D,V,T", [(8192, 4096, 128256, 2048), (4096, 5120, 152064, 1024)])
def test_full_vocabulary_ce_sampled_rows(L, D, V, T):
    """The Llama-3 vocabulary (V=128256, D=4096) and the 32B family's
    (V=152064, D=5120) in tiles of T rows: loss and dh rows against the
    oracle; one tile of all L rows gives identical bits for loss, dh and
    dW."""
    h, w, labels = synth.ce_inputs(L, D, V, device="cuda:0")
    scale = 1.0 / int((labels >= 0).sum())
    loss, dh, dw = upipe.ce_loss(h, w, labels, scale, T)
    torch.cuda.synchronize()
    status_ok()
    H, W = h.to("cpu", torch.float64).numpy(), w.to("cpu", torch.float64).numpy()
    lab = labels.cpu().numpy()
    rows = _rows(L, 6, 1)
    ml, mdh, _ = alst.ce_fwd_bwd(H[rows], W, lab[rows], scale, bf16_operands=True, weight_grad=False)
    assert_close(f64(loss[rows]), ml, "ce loss rows")
    assert_close(f64(dh[rows]), mdh, "ce dh rows")
    assert torch.isfinite(dw).all()
    loss1, dh1, dw1 = upipe.ce_loss(h, w, labels, scale, L)
    for a, b, n in zip((loss, dh, dw), (loss1, dh1, dw1), ("loss", "dh", "dW")):
        assert torch.equal(a, b), f"T={T} vs one tile: {n} differs"


def test_llama3_8b_mlp_and_loss_at_L2M():
    """The MLP and loss of a Llama-3-8B block at L = 2,097,152 tokens (the
    long-context sweep's largest length; D=4096, F=14336, V=128256).  Their
    untiled intermediates would need ~240 GB (MLP backward) and ~1.6 TB
    (fp32 logits and bf16 dZ) of device memory; tiles of T=16384 / 4096 rows
    hold 1.9 GB and 3.2 GB.  Sampled rows of y, dx, loss and dh against the
    precision-model oracle; every weight gradient finite."""
    L, D, F, V = 1 << 21, 4096, 14336, 128256
    Tm, Tc = 16384, 4096
    assert upipe.mlp_workspace_bytes(L, D, F, L, 1) > 200e9
    assert upipe.ce_workspace_bytes(L, D, V, L) > 1e12
    x, wgu, wd, dy = synth.mlp_inputs(L, D, F, device="cuda:0")
    y = upipe.mlp_forward(x, wgu, wd, Tm)
    dx, dwgu, dwd = upipe.mlp_backward(x, wgu, wd, dy, Tm)
    torch.cuda.synchronize()
    status_ok()
    rows = _rows(L, 8, 2)
    X, DY = (t[rows].to("cpu", torch.float64).numpy() for t in (x, dy))
    WGU, WD = (t.to("cpu", torch.float64).numpy() for t in (wgu, wd))
    my, _ = alst.mlp_fwd(X, WGU, WD, bf16_operands=True)
    mdx, _, _ = alst.mlp_bwd(X, WGU, WD, DY, bf16_operands=True, weight_grads=False)
    assert_close(f64(y[rows]), my, "mlp y rows (L=2M)")
    assert_close(f64(dx[rows]), mdx, "mlp dx rows (L=2M)")
    assert torch.isfinite(dwgu).all() and torch.isfinite(dwd).all()
    del y, dx, dwgu, dwd, dy, wgu, wd
    torch.cuda.empty_cache()
    _, w, labels = synth.ce_inputs(128, D, V, device="cuda:0")  # W only
    g = torch.Generator(device="cpu")
    g.manual_seed(23)
    labels = torch.randint(0, V, (L,), generator=g, dtype=torch.int32).to("cuda:0")
    scale = 1.0 / L
    loss, dh, dw = upipe.ce_loss(x, w, labels, scale, Tc)  # x serves as the final hidden states
    torch.cuda.synchronize()
    status_ok()
    W = w.to("cpu", torch.float64).numpy()
    ml, mdh, _ = alst.ce_fwd_bwd(X, W, labels[rows].cpu().numpy(), scale, bf16_operands=True, weight_grad=False)
    assert_close(f64(loss[rows]), ml, "ce loss rows (L=2M)")
    assert_close(f64(dh[rows]), mdh, "ce dh rows (L=2M)")
    assert torch.isfinite(loss).all() and torch.isfinite(dw).all()
