"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/upipe.h declares, plans workspaces by the stated
arithmetic and rejects bad arguments before touching a device."""

import ctypes
import os
import re

import pytest

from headwise_chunked_context_gb300 import upipe
from oracle import upipe_oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "upipe.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(upipe.LIB_PATH):
        from headwise_chunked_context_gb300 import build
        build.build()
    return upipe.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(upipe_[a-z_]+)\s*\(", text)))


def test_header_declares_what_binding_uses():
    assert declared_symbols() == sorted(upipe.EXPORTS)


def test_kernel_kinds_match_the_header():
    """upipe.KINDS names the UPIPE_KIND_* values in order, and its length is
    UPIPE_KIND_COUNT, so profile_read() labels every kind correctly."""
    text = open(HEADER).read()
    kinds = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define UPIPE_KIND_([A-Z0-9_]+) (\d+)", text)}
    count = kinds.pop("COUNT")
    assert count == len(upipe.KINDS)
    assert sorted(kinds.values()) == list(range(count))
    for name, value in kinds.items():
        words = set(name.lower().split("_"))
        assert words <= set(upipe.KINDS[value].split("_")) | {"attn", "gemm", "bwd", "fwd"}, (name, upipe.KINDS[value])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_strerror(lib):
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(upipe.strerror(code), str) and upipe.strerror(code)


def _cfg(**kw):
    base = dict(L=1024, D=1024, H=8, Hkv=2, U=2)
    base.update(kw)
    return upipe.Config(**base)


@pytest.mark.parametrize("bad", [
    dict(L=0), dict(H=6, Hkv=4), dict(U=3), dict(d=64), dict(causal=0), dict(D=1000),
    dict(H=8, Hkv=2, U=8, D=0), dict(rope_theta=0.0), dict(H=8, Hkv=4, U=4, L=-5),
    dict(H=96, Hkv=8, U=8),
])
def test_invalid_configs_have_no_workspace(lib, bad):
    assert upipe.workspace_bytes(_cfg(**bad), 0) == 0
    assert upipe.workspace_bytes(_cfg(**bad), 1) == 0


def test_u_not_a_multiple_or_divisor_of_group_is_rejected(lib):
    # H=12, Hkv=2 -> g=6; U=4 neither divides 6 nor is a multiple of it.
    assert upipe.workspace_bytes(_cfg(H=12, Hkv=2, U=4), 0) == 0
    assert upipe.workspace_bytes(_cfg(H=12, Hkv=2, U=3), 0) > 0
    assert upipe.workspace_bytes(_cfg(H=12, Hkv=2, U=12), 0) > 0


def test_entry_points_reject_bad_arguments_on_host(lib):
    c = _cfg().c()
    nullp = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: rejected first
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert lib.upipe_attn_fwd(ctypes.byref(c), nullp, fake, fake, fake, fake, None, fake, 1 << 40, None) == -1
    assert lib.upipe_attn_fwd(ctypes.byref(c), odd, fake, fake, fake, fake, None, fake, 1 << 40, None) == -1
    assert lib.upipe_attn_fwd(ctypes.byref(c), fake, fake, fake, fake, fake, None, fake, 16, None) == -2
    bad = _cfg(U=3).c()
    assert lib.upipe_attn_bwd(ctypes.byref(bad), fake, fake, fake, fake, fake, None, fake, fake, fake, fake,
                              1 << 40, None) == -1
    assert lib.upipe_attn_core_bwd(ctypes.byref(c), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                   0, None) == -2
    assert lib.upipe_attn_core_fwd(None, fake, fake, fake, fake, fake, None, 0, None) == -1


def test_workspace_arithmetic(lib):
    L, D, H, Hkv, U = 1024, 1024, 8, 2, 2
    c = _cfg()
    slot = L * 128 * 2
    al = lambda b: (b + 1023) // 1024 * 1024
    kvc = 1
    fwd = al(L * 64 * 8) + al((U + 2 * kvc) * slot) + al(U * slot) + al(L * D * 4)
    assert upipe.workspace_bytes(c, 0) == fwd
    assert upipe.workspace_bytes(c, 0, o_mode=upipe.O_DEVICE) == fwd - al(U * slot)
    # O in host memory: three chunk buffers of O in the forward, two in the
    # backward, in place of one
    assert upipe.workspace_bytes(c, 0, o_mode=upipe.O_HOST) == fwd - al(U * slot) + al(3 * U * slot)
    assert upipe.workspace_bytes(c, 0, o_mode=3) == 0 and upipe.workspace_bytes(c, 0, o_mode=-1) == 0
    rec = U * ((L + 63) // 64) * 128 * 4  # LSE/Delta records
    bwd = (al(L * 64 * 8) + al((U + 2 * kvc) * slot) + al(U * slot) + al(U * slot) + al(rec)
           + al(2 * (U + 2 * kvc) * slot) + al(2 * L * 128 * 4) + al(L * D * 4))
    assert upipe.workspace_bytes(c, 1) == bwd
    assert upipe.workspace_bytes(c, 1, o_mode=upipe.O_HOST) == bwd - al(U * slot) + al(2 * U * slot)
    # unchunked: no carries
    assert upipe.workspace_bytes(_cfg(U=8), 0) == al(L * 64 * 8) + al(12 * slot) + al(8 * slot)
    assert upipe.workspace_bytes(_cfg(), 0, core_only=True) == 0
    assert upipe.workspace_bytes(_cfg(), 1, core_only=True) == al(rec) + al(2 * L * 128 * 4)


@pytest.mark.parametrize("H,Hkv,L", [(32, 8, 32768), (64, 8, 131072), (32, 8, 65536)])
def test_chunk_memory_scales_as_u_over_h(lib, H, Hkv, L):
    D = 4096
    full_f, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=H), 0)
    full_b, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=H), 1)
    g = H // Hkv
    for U in [u for u in (g, 2 * g, H // 2) if H % u == 0 and u % g == 0]:
        f, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=U), 0)
        b, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=U), 1)
        assert f * H == full_f * U
        assert b * H == full_b * U
        # the forward chunk buffers are exactly the oracle's Q/K/V/O arithmetic
        assert f == orc.intermediate_bytes(L, U, H, Hkv, 128)


def test_32b_shape_u8_saves_87_5_percent(lib):
    L, D, H, Hkv = 131072, 5120, 64, 8
    full, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=64), 1)
    u8, _ = upipe.activation_bytes(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=8), 1)
    assert 1 - u8 / full == pytest.approx(0.875, abs=0)


# --------------------------------------------------------- chunk-size choice

def _valid_us(H, Hkv):
    g = H // Hkv
    return [u for u in range(1, H + 1) if H % u == 0 and (u % g == 0 or g % u == 0)]


def _need(cfg, pass_):
    if pass_ == 2:
        return max(upipe.workspace_bytes(cfg, 0), upipe.workspace_bytes(cfg, 1))
    return upipe.workspace_bytes(cfg, pass_)


@pytest.mark.parametrize("pass_", [0, 1, 2])
@pytest.mark.parametrize("L,D,H,Hkv", [(32768, 4096, 32, 8), (131072, 5120, 64, 8), (1024, 1024, 8, 2)])
def test_choose_u_is_the_largest_fitting_chunk(lib, pass_, L, D, H, Hkv):
    """At a budget equal to some U's workspace that U (or a larger one that
    also fits) is chosen; one byte less never yields it."""
    for u in _valid_us(H, Hkv):
        cfg = upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=u)
        need = _need(cfg, pass_)
        fits = [v for v in _valid_us(H, Hkv) if _need(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=v), pass_) <= need]
        assert upipe.choose_u(cfg, need, pass_) == max(fits)
        below = [v for v in _valid_us(H, Hkv) if _need(upipe.Config(L=L, D=D, H=H, Hkv=Hkv, U=v), pass_) < need]
        if below:
            assert upipe.choose_u(cfg, need - 1, pass_) == max(below)


def test_choose_u_budget_below_every_chunk_size(lib):
    cfg = upipe.Config(L=32768, D=4096, H=32, Hkv=8, U=8)
    smallest = min(_need(upipe.Config(L=32768, D=4096, H=32, Hkv=8, U=u), 2) for u in _valid_us(32, 8))
    with pytest.raises(upipe.UpipeError) as e:
        upipe.choose_u(cfg, smallest - 1)
    assert e.value.code == upipe.UPIPE_ERR_WS_TOO_SMALL
    assert upipe.choose_u(cfg, 1 << 62) == 32  # unlimited: the unchunked layer


def test_choose_u_ignores_cfg_u_and_rejects_bad_arguments(lib):
    a = upipe.Config(L=8192, D=4096, H=32, Hkv=8, U=3)  # U itself invalid: ignored
    b = upipe.Config(L=8192, D=4096, H=32, Hkv=8, U=8)
    budget = upipe.workspace_bytes(b, 1)
    assert upipe.choose_u(a, budget, 1) == upipe.choose_u(b, budget, 1)
    c = upipe.Config(L=8192, D=4096, H=32, Hkv=8, U=8).c()
    assert lib.upipe_choose_u(ctypes.byref(c), 1 << 40, 3, 0, 0) == upipe.UPIPE_ERR_INVALID_ARG
    assert lib.upipe_choose_u(None, 1 << 40, 2, 0, 0) == upipe.UPIPE_ERR_INVALID_ARG
    bad = upipe.Config(L=8192, D=4096, H=30, Hkv=8, U=8).c()
    assert lib.upipe_choose_u(ctypes.byref(bad), 1 << 40, 2, 0, 0) == upipe.UPIPE_ERR_INVALID_ARG


def test_choose_u_picks_u8_for_the_32b_layer_at_its_workspace(lib):
    """The 32B-shaped layer (L=131072): a budget of U=8's training-step
    workspace selects U=8 (U=16 needs more)."""
    cfg = upipe.Config(L=131072, D=5120, H=64, Hkv=8, U=8)
    assert upipe.choose_u(cfg, _need(cfg, 2), 2) == 8


# ------------------------------------------- argument checks of the binding

def test_binding_rejects_mis_shaped_or_mis_typed_tensors_before_any_launch(lib):
    """Shapes and dtypes of every tensor argument are checked in Python
    before the library is called (CPU tensors: nothing can launch)."""
    import torch
    cfg = upipe.Config(L=64, H=4, Hkv=2, U=2)
    q = torch.zeros(64, 4, 128, dtype=torch.bfloat16)
    k = torch.zeros(64, 2, 128, dtype=torch.bfloat16)
    lse = torch.zeros(4, 64, dtype=torch.float32)
    n0 = upipe.launch_count()
    short_q = torch.zeros(63, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q"):
        upipe.attn_core_bwd(cfg, short_q, k, k, q, lse, q, q, k, k)
    with pytest.raises(ValueError, match="lse"):
        upipe.attn_core_bwd(cfg, q, k, k, q, lse[:, :32], q, q, k, k)
    with pytest.raises(ValueError, match="o"):
        upipe.attn_core_bwd_noalloc(cfg, q, k, k, q.float(), lse, q, q, k, k)
    with pytest.raises(ValueError, match="v"):
        upipe.attn_core_fwd(cfg, q, k, torch.zeros(64, 1, 128, dtype=torch.bfloat16), q, lse)
    with pytest.raises(ValueError, match="CUDA"):
        upipe.attn_core_fwd(cfg, q, k, k, q, lse)
    lcfg = upipe.Config(L=64, D=256, H=4, Hkv=2, U=2)
    x = torch.zeros(64, 256, dtype=torch.bfloat16)
    w = torch.zeros(8 * 128, 256, dtype=torch.bfloat16)
    wo = torch.zeros(256, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="x"):
        upipe.attn_bwd(lcfg, x[:32], w, wo, x, lse, x, w.float(), wo.float())
    with pytest.raises(ValueError, match="Wo"):
        upipe.attn_bwd(lcfg, x, w, wo.t(), x, lse, x, w.float(), wo.float())
    with pytest.raises(ValueError, match="o_saved"):
        upipe.attn_bwd(lcfg, x, w, wo, x, lse, x, w.float(), wo.float(), o_saved=x)
    with pytest.raises(ValueError, match="Wqkv"):
        upipe.attn_fwd(lcfg, x, w[:512], wo, x, lse)
    assert upipe.launch_count() == n0


def test_offload_entry_points_reject_null_buffers_before_any_copy(lib):
    """A zero-byte copy is a no-op and a null buffer with bytes > 0 is an
    argument error; neither reaches the CUDA runtime."""
    assert lib.upipe_prefetch_async(None, None, 0, None) == upipe.UPIPE_OK
    assert lib.upipe_prefetch_async(None, ctypes.c_void_p(1 << 20), 64, None) == upipe.UPIPE_ERR_INVALID_ARG
    assert lib.upipe_offload_async(ctypes.c_void_p(1 << 20), None, 64, None) == upipe.UPIPE_ERR_INVALID_ARG


def test_host_o_entry_points_reject_null_or_unpinned_buffers(lib):
    """O kept in host memory must be page-locked: a null o_host is an
    argument error in the library, a pageable or mis-sized tensor in the
    binding; nothing is launched."""
    import torch
    c = _cfg().c()
    fake = ctypes.c_void_p(1 << 20)
    n0 = upipe.launch_count()
    assert lib.upipe_attn_fwd_host_o(ctypes.byref(c), fake, fake, fake, fake, fake, None, fake, 1 << 30,
                                     None) == upipe.UPIPE_ERR_INVALID_ARG
    assert lib.upipe_attn_bwd_host_o(ctypes.byref(c), fake, fake, fake, fake, fake, None, fake, fake, fake, fake,
                                     1 << 30, None) == upipe.UPIPE_ERR_INVALID_ARG
    cfg = upipe.Config(L=256, D=256, H=4, Hkv=2, U=2)
    x = torch.zeros(256, 256, dtype=torch.bfloat16)
    w = torch.zeros(8 * 128, 256, dtype=torch.bfloat16)
    wo = torch.zeros(256, 512, dtype=torch.bfloat16)
    lse = torch.zeros(4, 256)
    with pytest.raises(ValueError, match="o_host"):
        upipe.attn_fwd_host_o(cfg, x, w, wo, x, lse, torch.zeros(256 * 512, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="o_host"):
        upipe.attn_fwd_host_o(cfg, x, w, wo, x, lse, torch.zeros(7, dtype=torch.bfloat16))
    assert upipe.launch_count() == n0


# ----------------------------------------- sequence-tiled MLP and loss (host)

def test_tiled_mlp_and_loss_workspace_scales_with_the_tile(lib):
    """The MLP keeps one tile's H [T, F] (forward) or H, dH and dG|dU
    (backward) and the loss one tile's fp32 logits and bf16 dZ [T, V]: the
    workspace is proportional to T and independent of L."""
    al = lambda b: (b + 1023) // 1024 * 1024
    D, F, V = 4096, 14336, 128256
    for T in (1024, 8192):
        tf = T * F * 2
        assert upipe.mlp_workspace_bytes(1 << 20, D, F, T, 0) == al(tf)
        assert upipe.mlp_workspace_bytes(1 << 20, D, F, T, 1) == al(tf) * 2 + al(2 * tf)
        assert upipe.mlp_workspace_bytes(3 << 20, D, F, T, 1) == upipe.mlp_workspace_bytes(1 << 20, D, F, T, 1)
        assert upipe.ce_workspace_bytes(1 << 20, D, V, T) == al(T * V * 4) + al(T * V * 2)
    assert upipe.mlp_workspace_bytes(1 << 20, D, F, 8192, 1) == 8 * upipe.mlp_workspace_bytes(1 << 20, D, F, 1024, 1)
    # the oracle's own accounting of one tile's intermediates agrees
    assert upipe.mlp_workspace_bytes(1 << 20, D, F, 8192, 1) == orc_alst().tile_bytes(8192, D, F, V)["mlp_bwd"]
    assert upipe.ce_workspace_bytes(1 << 20, D, V, 8192) == orc_alst().tile_bytes(8192, D, F, V)["ce"]


def orc_alst():
    from oracle import alst_oracle
    return alst_oracle


@pytest.mark.parametrize("L,D,F,T", [(0, 256, 256, 128), (100, 100, 256, 128), (100, 256, 200, 128),
                                     (100, 256, 256, 100), (100, 256, 256, 0)])
def test_tiled_mlp_rejects_bad_shapes(lib, L, D, F, T):
    assert upipe.mlp_workspace_bytes(L, D, F, T, 1) == 0
    assert upipe.ce_workspace_bytes(L, D, F, T) == 0  # V takes F's place: same constraints
    c = upipe.MlpCfg(L, D, F, T)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.upipe_mlp_fwd(ctypes.byref(c), fake, fake, fake, fake, fake, 1 << 30, None) == upipe.UPIPE_ERR_INVALID_ARG


def test_tiled_entry_points_reject_null_pointers_before_any_launch(lib):
    n0 = upipe.launch_count()
    m = upipe.MlpCfg(1024, 256, 512, 256)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.upipe_mlp_fwd(ctypes.byref(m), fake, None, fake, fake, fake, 1 << 30, None) == -1
    assert lib.upipe_mlp_bwd(ctypes.byref(m), fake, fake, fake, fake, fake, fake, None, fake, 1 << 30, None) == -1
    assert lib.upipe_mlp_fwd(ctypes.byref(m), fake, fake, fake, fake, fake, 16, None) == upipe.UPIPE_ERR_WS_TOO_SMALL
    c = upipe.CeCfg(1024, 256, 512, 256)
    assert lib.upipe_ce_fwd_bwd(ctypes.byref(c), fake, fake, None, ctypes.c_float(1.0), fake, fake, fake, fake,
                                1 << 32, None) == -1
    assert lib.upipe_ce_fwd_bwd(ctypes.byref(c), fake, fake, fake, ctypes.c_float(float("inf")), fake, fake, fake,
                                fake, 1 << 32, None) == -1
    assert upipe.launch_count() == n0


@pytest.mark.parametrize("L,D,F,V", [(131072, 5120, 27648, 152064), (1000, 256, 512, 1024), (100, 128, 128, 128)])
def test_tile_from_a_memory_budget(lib, L, D, F, V):
    """The largest tile whose workspace fits: at a budget equal to some T's
    bytes that T is chosen, one byte less gives the T below it; never more
    than L rounded up to 128; below T = 128's bytes it is an error."""
    t_max = (L + 127) // 128 * 128
    for T in sorted({128, min(t_max, 1024), t_max}):
        for pass_ in (0, 1):
            need = upipe.mlp_workspace_bytes(L, D, F, T, pass_)
            assert upipe.mlp_choose_t(L, D, F, need, pass_) == T
            if T > 128:
                assert upipe.mlp_choose_t(L, D, F, need - 1, pass_) == T - 128
        need = upipe.ce_workspace_bytes(L, D, V, T)
        assert upipe.ce_choose_t(L, D, V, need) == T
        if T > 128:
            assert upipe.ce_choose_t(L, D, V, need - 1) == T - 128
    assert upipe.mlp_choose_t(L, D, F, 1 << 62) == t_max
    assert upipe.ce_choose_t(L, D, V, 1 << 62) == t_max
    assert upipe.mlp_choose_t(L, D, F, upipe.mlp_workspace_bytes(L, D, F, 128, 1), 2) == 128
    with pytest.raises(upipe.UpipeError):
        upipe.mlp_choose_t(L, D, F, upipe.mlp_workspace_bytes(L, D, F, 128, 1) - 1, 1)
    with pytest.raises(upipe.UpipeError):
        upipe.ce_choose_t(L, D, V, 1000)
    with pytest.raises(upipe.UpipeError):
        upipe.mlp_choose_t(L, 100, F, 1 << 40)
