"""Thin ctypes binding of libupipe.so (declared in include/upipe.h).

Argument marshalling only: torch tensors are checked for dtype, shape,
device and contiguity, then their device pointers and the current CUDA
stream are handed to the C entry points of the same names.  Every step of
the attention layer runs in the library's sm_103a kernels; there is no
fallback path, and a missing library raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libupipe.so")

UPIPE_OK = 0
UPIPE_ERR_INVALID_ARG = -1
UPIPE_ERR_WS_TOO_SMALL = -2
UPIPE_ERR_CUDA = -3
UPIPE_ERR_DEVICE_TIMEOUT = -4
UPIPE_ERR_UNSUPPORTED_DEVICE = -5
UPIPE_ERR_SCRATCH_LIMIT = -6
NOALLOC_SCRATCH_BYTES = 32 << 20
O_RECOMPUTE, O_DEVICE, O_HOST = 0, 1, 2  # where the layer keeps O between forward and backward

EXPORTS = (
    "upipe_workspace_bytes",
    "upipe_activation_bytes",
    "upipe_choose_u",
    "upipe_attn_fwd",
    "upipe_attn_bwd",
    "upipe_attn_fwd_host_o",
    "upipe_attn_bwd_host_o",
    "upipe_attn_core_fwd",
    "upipe_attn_core_bwd",
    "upipe_attn_core_bwd_noalloc",
    "upipe_mlp_workspace_bytes",
    "upipe_mlp_fwd",
    "upipe_mlp_bwd",
    "upipe_ce_workspace_bytes",
    "upipe_ce_fwd_bwd",
    "upipe_mlp_choose_t",
    "upipe_ce_choose_t",
    "upipe_offload_async",
    "upipe_prefetch_async",
    "upipe_copies_join",
    "upipe_last_device_status",
    "upipe_debug_wait_timeout",
    "upipe_launch_count",
    "upipe_profile_enable",
    "upipe_profile_read",
    "upipe_strerror",
)

KINDS = ("rope_table", "qkv_gemm", "attn_fwd", "oproj_gemm", "do_gemm", "dwo_gemm", "attn_bwd_dq",
         "attn_bwd_dkdv", "dwqkv_gemm", "dx_gemm", "delta", "zero_rows", "alst_gu", "alst_gemm", "alst_wgrad",
         "ce_rows")


class UpipeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class Cfg(ctypes.Structure):
    """Mirror of ``upipe_cfg``."""

    _fields_ = [
        ("L", ctypes.c_int64),
        ("D", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("U", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("rope_theta", ctypes.c_double),
    ]


class MlpCfg(ctypes.Structure):
    """Mirror of ``upipe_mlp_cfg``."""

    _fields_ = [("L", ctypes.c_int64), ("D", ctypes.c_int32), ("F", ctypes.c_int32), ("T", ctypes.c_int32)]


class CeCfg(ctypes.Structure):
    """Mirror of ``upipe_ce_cfg``."""

    _fields_ = [("L", ctypes.c_int64), ("D", ctypes.c_int32), ("V", ctypes.c_int32), ("T", ctypes.c_int32)]


@dataclass(frozen=True)
class Config:
    L: int
    H: int
    Hkv: int
    U: int
    D: int = 0
    d: int = 128
    rope_theta: float = 500000.0
    causal: int = 1

    def c(self) -> Cfg:
        return Cfg(self.L, self.D, self.H, self.Hkv, self.d, self.U, self.causal, self.rope_theta)


_lib = None


def lib() -> ctypes.CDLL:
    """Opens libupipe.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with headwise_chunked_context_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        cfgp = ctypes.POINTER(Cfg)
        L.upipe_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_workspace_bytes.argtypes = [cfgp, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.upipe_activation_bytes.restype = ctypes.c_int
        L.upipe_activation_bytes.argtypes = [cfgp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
        L.upipe_choose_u.restype = ctypes.c_int
        L.upipe_choose_u.argtypes = [cfgp, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.upipe_attn_fwd.restype = ctypes.c_int
        L.upipe_attn_fwd.argtypes = [cfgp, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_bwd.restype = ctypes.c_int
        L.upipe_attn_bwd.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_fwd_host_o.restype = ctypes.c_int
        L.upipe_attn_fwd_host_o.argtypes = [cfgp, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_bwd_host_o.restype = ctypes.c_int
        L.upipe_attn_bwd_host_o.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_core_fwd.restype = ctypes.c_int
        L.upipe_attn_core_fwd.argtypes = [cfgp, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_core_bwd.restype = ctypes.c_int
        L.upipe_attn_core_bwd.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_attn_core_bwd_noalloc.restype = ctypes.c_int
        L.upipe_attn_core_bwd_noalloc.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, P]
        mcfg, ccfg = ctypes.POINTER(MlpCfg), ctypes.POINTER(CeCfg)
        L.upipe_mlp_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_mlp_workspace_bytes.argtypes = [mcfg, ctypes.c_int]
        L.upipe_mlp_fwd.restype = ctypes.c_int
        L.upipe_mlp_fwd.argtypes = [mcfg, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_mlp_bwd.restype = ctypes.c_int
        L.upipe_mlp_bwd.argtypes = [mcfg, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_ce_workspace_bytes.restype = ctypes.c_size_t
        L.upipe_ce_workspace_bytes.argtypes = [ccfg]
        L.upipe_mlp_choose_t.restype = ctypes.c_int
        L.upipe_mlp_choose_t.argtypes = [mcfg, ctypes.c_size_t, ctypes.c_int]
        L.upipe_ce_choose_t.restype = ctypes.c_int
        L.upipe_ce_choose_t.argtypes = [ccfg, ctypes.c_size_t]
        L.upipe_ce_fwd_bwd.restype = ctypes.c_int
        L.upipe_ce_fwd_bwd.argtypes = [ccfg, P, P, P, ctypes.c_float, P, P, P, P, ctypes.c_size_t, P]
        L.upipe_offload_async.restype = ctypes.c_int
        L.upipe_offload_async.argtypes = [P, P, ctypes.c_size_t, P]
        L.upipe_prefetch_async.restype = ctypes.c_int
        L.upipe_prefetch_async.argtypes = [P, P, ctypes.c_size_t, P]
        L.upipe_copies_join.restype = ctypes.c_int
        L.upipe_copies_join.argtypes = [P]
        L.upipe_last_device_status.restype = ctypes.c_int
        L.upipe_last_device_status.argtypes = [P]
        L.upipe_debug_wait_timeout.restype = ctypes.c_int
        L.upipe_debug_wait_timeout.argtypes = [ctypes.c_uint64, P]
        L.upipe_launch_count.restype = ctypes.c_int64
        L.upipe_launch_count.argtypes = []
        L.upipe_profile_enable.restype = None
        L.upipe_profile_enable.argtypes = [ctypes.c_int]
        L.upipe_profile_read.restype = ctypes.c_int
        L.upipe_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                         ctypes.c_int]
        L.upipe_strerror.restype = ctypes.c_char_p
        L.upipe_strerror.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().upipe_strerror(code).decode()


def _check(code: int, where: str) -> None:
    if code != UPIPE_OK:
        raise UpipeError(code, where)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _expect(t, shape, dtype, name):
    """Checks one tensor argument's shape and dtype before anything reaches
    the library: the kernels read and write exactly the sizes the
    configuration implies, so a smaller tensor must be refused here."""
    if t is None:
        raise ValueError(f"{name}: missing")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")


def _on_device(**tensors):
    """Every tensor argument must be a contiguous CUDA tensor on the current
    device (the kernels run there and take raw pointers)."""
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name}: expected a CUDA tensor, got one on {t.device}")
        if t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
        if not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous tensor")


def _expect_ws(ws, need, name="ws"):
    if ws is None:
        return
    _on_device(**{name: ws})
    if ws.numel() * ws.element_size() < need:
        raise ValueError(f"{name}: {ws.numel() * ws.element_size()} bytes, the call needs {need}")


# ----------------------------------------------------------- raw entry points

def workspace_bytes(cfg: Config, pass_: int, core_only: bool = False, o_mode: int = O_RECOMPUTE) -> int:
    """o_mode: O_RECOMPUTE, O_DEVICE (o_saved given) or O_HOST (the _host_o
    entries); True / False read as O_DEVICE / O_RECOMPUTE."""
    c = cfg.c()
    return int(lib().upipe_workspace_bytes(ctypes.byref(c), pass_, int(core_only), int(o_mode)))


def activation_bytes(cfg: Config, pass_: int, core_only: bool = False, o_mode: int = O_RECOMPUTE):
    c = cfg.c()
    chunk = ctypes.c_size_t(0)
    fixed = ctypes.c_size_t(0)
    _check(lib().upipe_activation_bytes(ctypes.byref(c), pass_, int(core_only), int(o_mode),
                                        ctypes.byref(chunk), ctypes.byref(fixed)), "upipe_activation_bytes")
    return int(chunk.value), int(fixed.value)


def choose_u(cfg: Config, budget_bytes: int, pass_: int = 2, core_only: bool = False,
             o_mode: int = O_RECOMPUTE) -> int:
    """Largest valid chunk size U whose workspace fits `budget_bytes`
    (upipe_choose_u; cfg.U is ignored).  pass_ 0 = forward, 1 = backward,
    2 = the larger of the two.  Raises UpipeError when no U fits."""
    c = cfg.c()
    r = int(lib().upipe_choose_u(ctypes.byref(c), int(budget_bytes), pass_, int(core_only), int(o_mode)))
    if r < 0:
        raise UpipeError(r, "upipe_choose_u")
    return r


def _ws(cfg, pass_, core_only, o_mode, ws, device):
    need = workspace_bytes(cfg, pass_, core_only, o_mode)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    _expect_ws(ws, need)
    return ws, ws.numel() * ws.element_size()


def _layer_tensors(cfg: Config, x, Wqkv, Wo, lse, o_saved):
    L, D, H, Hkv = cfg.L, cfg.D, cfg.H, cfg.Hkv
    _expect(x, (L, D), torch.bfloat16, "x")
    _expect(Wqkv, ((H + 2 * Hkv) * 128, D), torch.bfloat16, "Wqkv")
    _expect(Wo, (D, H * 128), torch.bfloat16, "Wo")
    _expect(lse, (H, L), torch.float32, "lse")
    if o_saved is not None:
        _expect(o_saved, (L, H * 128), torch.bfloat16, "o_saved")


def _core_tensors(cfg: Config, q, k, v, lse, o=None):
    L, H, Hkv = cfg.L, cfg.H, cfg.Hkv
    _expect(q, (L, H, 128), torch.bfloat16, "q")
    _expect(k, (L, Hkv, 128), torch.bfloat16, "k")
    _expect(v, (L, Hkv, 128), torch.bfloat16, "v")
    _expect(lse, (H, L), torch.float32, "lse")
    if o is not None:
        _expect(o, (L, H, 128), torch.bfloat16, "o")


def _core_grads(cfg: Config, do, dq, dk, dv):
    L, H, Hkv = cfg.L, cfg.H, cfg.Hkv
    for t, shp, n in ((do, (L, H, 128), "dout_o"), (dq, (L, H, 128), "dq"), (dk, (L, Hkv, 128), "dk"),
                      (dv, (L, Hkv, 128), "dv")):
        _expect(t, shp, torch.bfloat16, n)


def attn_fwd(cfg: Config, x, Wqkv, Wo, out, lse, o_saved=None, ws=None, stream=None):
    _layer_tensors(cfg, x, Wqkv, Wo, lse, o_saved)
    _expect(out, (cfg.L, cfg.D), torch.bfloat16, "out")
    _on_device(x=x, Wqkv=Wqkv, Wo=Wo, out=out, lse=lse, o_saved=o_saved)
    ws, nbytes = _ws(cfg, 0, False, O_DEVICE if o_saved is not None else O_RECOMPUTE, ws, x.device)
    c = cfg.c()
    _check(lib().upipe_attn_fwd(ctypes.byref(c), _ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(out), _ptr(lse),
                                _ptr(o_saved), _ptr(ws), nbytes, _stream(stream)), "upipe_attn_fwd")


def attn_bwd(cfg: Config, x, Wqkv, Wo, dout, lse, dx, dWqkv, dWo, o_saved=None, ws=None, stream=None):
    L, D, H, Hkv = cfg.L, cfg.D, cfg.H, cfg.Hkv
    _layer_tensors(cfg, x, Wqkv, Wo, lse, o_saved)
    _expect(dout, (L, D), torch.bfloat16, "dout")
    _expect(dx, (L, D), torch.bfloat16, "dx")
    _expect(dWqkv, ((H + 2 * Hkv) * 128, D), torch.float32, "dWqkv")
    _expect(dWo, (D, H * 128), torch.float32, "dWo")
    _on_device(x=x, Wqkv=Wqkv, Wo=Wo, dout=dout, lse=lse, o_saved=o_saved, dx=dx, dWqkv=dWqkv, dWo=dWo)
    ws, nbytes = _ws(cfg, 1, False, O_DEVICE if o_saved is not None else O_RECOMPUTE, ws, x.device)
    c = cfg.c()
    _check(lib().upipe_attn_bwd(ctypes.byref(c), _ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(dout), _ptr(lse),
                                _ptr(o_saved), _ptr(dx), _ptr(dWqkv), _ptr(dWo), _ptr(ws), nbytes,
                                _stream(stream)), "upipe_attn_bwd")


def _host_o(cfg: Config, o_host):
    """o_host: a page-locked CPU tensor of L*H*128 bf16 (any shape)."""
    if o_host is None:
        raise ValueError("o_host: missing")
    if o_host.is_cuda or o_host.dtype != torch.bfloat16 or o_host.numel() != cfg.L * cfg.H * 128:
        raise ValueError(f"o_host: expected {cfg.L * cfg.H * 128} bf16 elements in host memory, got "
                         f"{o_host.numel()} {o_host.dtype} on {o_host.device}")
    if not o_host.is_contiguous() or not o_host.is_pinned():
        raise ValueError("o_host: expected a contiguous page-locked (pinned) tensor")
    return ctypes.c_void_p(o_host.data_ptr())


def new_host_o(cfg: Config):
    """Page-locked host buffer for upipe_attn_fwd_host_o: chunk c's O_c
    [L, U*128] at element offset c*L*U*128."""
    return torch.empty((cfg.H // cfg.U, cfg.L, cfg.U * 128), dtype=torch.bfloat16, pin_memory=True)


def attn_fwd_host_o(cfg: Config, x, Wqkv, Wo, out, lse, o_host, ws=None, stream=None):
    _layer_tensors(cfg, x, Wqkv, Wo, lse, None)
    _expect(out, (cfg.L, cfg.D), torch.bfloat16, "out")
    oh = _host_o(cfg, o_host)
    _on_device(x=x, Wqkv=Wqkv, Wo=Wo, out=out, lse=lse)
    ws, nbytes = _ws(cfg, 0, False, O_HOST, ws, x.device)
    c = cfg.c()
    _check(lib().upipe_attn_fwd_host_o(ctypes.byref(c), _ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(out), _ptr(lse),
                                       oh, _ptr(ws), nbytes, _stream(stream)), "upipe_attn_fwd_host_o")


def attn_bwd_host_o(cfg: Config, x, Wqkv, Wo, dout, lse, o_host, dx, dWqkv, dWo, ws=None, stream=None):
    L, D, H, Hkv = cfg.L, cfg.D, cfg.H, cfg.Hkv
    _layer_tensors(cfg, x, Wqkv, Wo, lse, None)
    _expect(dout, (L, D), torch.bfloat16, "dout")
    _expect(dx, (L, D), torch.bfloat16, "dx")
    _expect(dWqkv, ((H + 2 * Hkv) * 128, D), torch.float32, "dWqkv")
    _expect(dWo, (D, H * 128), torch.float32, "dWo")
    oh = _host_o(cfg, o_host)
    _on_device(x=x, Wqkv=Wqkv, Wo=Wo, dout=dout, lse=lse, dx=dx, dWqkv=dWqkv, dWo=dWo)
    ws, nbytes = _ws(cfg, 1, False, O_HOST, ws, x.device)
    c = cfg.c()
    _check(lib().upipe_attn_bwd_host_o(ctypes.byref(c), _ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(dout), _ptr(lse),
                                       oh, _ptr(dx), _ptr(dWqkv), _ptr(dWo), _ptr(ws), nbytes,
                                       _stream(stream)), "upipe_attn_bwd_host_o")


def attn_core_fwd(cfg: Config, q, k, v, o, lse, ws=None, stream=None):
    _core_tensors(cfg, q, k, v, lse, o)
    _on_device(q=q, k=k, v=v, o=o, lse=lse)
    need = workspace_bytes(cfg, 0, True)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if need and ws is None:
        ws, nbytes = _ws(cfg, 0, True, False, None, q.device)
    _expect_ws(ws, need)
    c = cfg.c()
    _check(lib().upipe_attn_core_fwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                     _ptr(ws), nbytes, _stream(stream)), "upipe_attn_core_fwd")


def attn_core_bwd(cfg: Config, q, k, v, o, lse, do, dq, dk, dv, ws=None, stream=None):
    _core_tensors(cfg, q, k, v, lse, o)
    _core_grads(cfg, do, dq, dk, dv)
    _on_device(q=q, k=k, v=v, o=o, lse=lse, dout_o=do, dq=dq, dk=dk, dv=dv)
    ws, nbytes = _ws(cfg, 1, True, False, ws, q.device)
    c = cfg.c()
    _check(lib().upipe_attn_core_bwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), nbytes, _stream(stream)),
           "upipe_attn_core_bwd")


def attn_core_bwd_noalloc(cfg: Config, q, k, v, o, lse, do, dq, dk, dv, stream=None):
    """Core backward through the entry point that allocates nothing (its
    scratch is a fixed array in the library's static device memory; see
    include/upipe.h).  For callers that may not allocate at call time."""
    _core_tensors(cfg, q, k, v, lse, o)
    _core_grads(cfg, do, dq, dk, dv)
    _on_device(q=q, k=k, v=v, o=o, lse=lse, dout_o=do, dq=dq, dk=dk, dv=dv)
    c = cfg.c()
    _check(lib().upipe_attn_core_bwd_noalloc(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)),
           "upipe_attn_core_bwd_noalloc")


def _host_pair(host, devt, name):
    if host.is_cuda or not devt.is_cuda:
        raise ValueError(f"{name}: expected a host tensor and a CUDA tensor")
    if tuple(host.shape) != tuple(devt.shape) or host.dtype != devt.dtype:
        raise ValueError(f"{name}: host {tuple(host.shape)} {host.dtype} vs device {tuple(devt.shape)} {devt.dtype}")
    if not host.is_contiguous() or not devt.is_contiguous():
        raise ValueError(f"{name}: expected contiguous tensors")
    _on_device(**{name: devt})
    return devt.numel() * devt.element_size()


def offload_async(host, dev_tensor, stream=None) -> None:
    """Copies `dev_tensor` into the host tensor `host` (pinned for an
    asynchronous copy) on the library's copy stream, after the work already
    on `stream` (upipe_offload_async).  Call copies_join before reusing or
    releasing `dev_tensor`."""
    n = _host_pair(host, dev_tensor, "offload")
    _check(lib().upipe_offload_async(ctypes.c_void_p(host.data_ptr()), ctypes.c_void_p(dev_tensor.data_ptr()), n,
                                     _stream(stream)), "upipe_offload_async")


def prefetch_async(dev_tensor, host, stream=None) -> None:
    """Copies the host tensor `host` into `dev_tensor` on the library's copy
    stream, after the work already on `stream` (upipe_prefetch_async).  Call
    copies_join before using `dev_tensor`."""
    n = _host_pair(host, dev_tensor, "prefetch")
    _check(lib().upipe_prefetch_async(ctypes.c_void_p(dev_tensor.data_ptr()), ctypes.c_void_p(host.data_ptr()), n,
                                      _stream(stream)), "upipe_prefetch_async")


def copies_join(stream=None) -> None:
    """Work enqueued on `stream` afterwards waits for every offload and
    prefetch issued so far on the current device (upipe_copies_join)."""
    _check(lib().upipe_copies_join(_stream(stream)), "upipe_copies_join")


def last_device_status(stream=None) -> int:
    return int(lib().upipe_last_device_status(_stream(stream)))


def debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib().upipe_debug_wait_timeout(limit_ns, _stream(stream)), "upipe_debug_wait_timeout")


def launch_count() -> int:
    return int(lib().upipe_launch_count())


def profile_enable(on: bool) -> None:
    lib().upipe_profile_enable(int(on))


def profile_read():
    """{kind: (total ms, launches)} for launches recorded since the last read."""
    n = len(KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    lib().upipe_profile_read(ms, cnt, n)
    return {KINDS[k]: (float(ms[k]), int(cnt[k])) for k in range(n)}


# ------------------------------------------------------- allocating helpers

def layer_forward(cfg: Config, x, Wqkv, Wo, keep_o=False):
    """Allocates out [L, D] bf16, lse [H, L] fp32 and runs the layer forward.
    keep_o: False (O recomputed by the backward), True (O kept on the
    device, upipe_attn_fwd's o_saved) or "host" (O kept in page-locked host
    memory, upipe_attn_fwd_host_o).  Returns (out, lse, kept O or None)."""
    dev = x.device
    out = torch.empty((cfg.L, cfg.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((cfg.H, cfg.L), dtype=torch.float32, device=dev)
    if keep_o == "host":
        o_host = new_host_o(cfg)
        attn_fwd_host_o(cfg, x, Wqkv, Wo, out, lse, o_host)
        return out, lse, o_host
    o_saved = torch.empty((cfg.L, cfg.H * 128), dtype=torch.bfloat16, device=dev) if keep_o else None
    attn_fwd(cfg, x, Wqkv, Wo, out, lse, o_saved)
    return out, lse, o_saved


def layer_backward(cfg: Config, x, Wqkv, Wo, dout, lse, o_saved=None):
    """Allocates dx [L, D] bf16, dWqkv, dWo fp32 and runs the layer backward
    with the O that layer_forward kept (a host tensor selects
    upipe_attn_bwd_host_o)."""
    dev = x.device
    dx = torch.empty((cfg.L, cfg.D), dtype=torch.bfloat16, device=dev)
    dWqkv = torch.empty(((cfg.H + 2 * cfg.Hkv) * 128, cfg.D), dtype=torch.float32, device=dev)
    dWo = torch.empty((cfg.D, cfg.H * 128), dtype=torch.float32, device=dev)
    if o_saved is not None and not o_saved.is_cuda:
        attn_bwd_host_o(cfg, x, Wqkv, Wo, dout, lse, o_saved, dx, dWqkv, dWo)
    else:
        attn_bwd(cfg, x, Wqkv, Wo, dout, lse, dx, dWqkv, dWo, o_saved)
    return dx, dWqkv, dWo


def core_forward(cfg: Config, q, k, v):
    o = torch.empty_like(q)
    lse = torch.empty((cfg.H, cfg.L), dtype=torch.float32, device=q.device)
    attn_core_fwd(cfg, q, k, v, o, lse)
    return o, lse


def core_backward(cfg: Config, q, k, v, o, lse, do):
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    attn_core_bwd(cfg, q, k, v, o, lse, do, dq, dk, dv)
    return dq, dk, dv


# ------------------------------------------- sequence-tiled MLP and loss

def mlp_workspace_bytes(L: int, D: int, F: int, T: int, pass_: int) -> int:
    c = MlpCfg(L, D, F, T)
    return int(lib().upipe_mlp_workspace_bytes(ctypes.byref(c), pass_))


def mlp_choose_t(L: int, D: int, F: int, budget_bytes: int, pass_: int = 2) -> int:
    """Largest tile T whose MLP workspace fits the budget (upipe_mlp_choose_t)."""
    c = MlpCfg(L, D, F, 128)
    r = int(lib().upipe_mlp_choose_t(ctypes.byref(c), int(budget_bytes), pass_))
    if r < 0:
        raise UpipeError(r, "upipe_mlp_choose_t")
    return r


def ce_choose_t(L: int, D: int, V: int, budget_bytes: int) -> int:
    """Largest tile T whose loss workspace fits the budget (upipe_ce_choose_t)."""
    c = CeCfg(L, D, V, 128)
    r = int(lib().upipe_ce_choose_t(ctypes.byref(c), int(budget_bytes)))
    if r < 0:
        raise UpipeError(r, "upipe_ce_choose_t")
    return r


def ce_workspace_bytes(L: int, D: int, V: int, T: int) -> int:
    c = CeCfg(L, D, V, T)
    return int(lib().upipe_ce_workspace_bytes(ctypes.byref(c)))


def _tile_ws(need, ws, device):
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
    _expect_ws(ws, need)
    return ws, ws.numel() * ws.element_size()


def mlp_fwd(x, Wgu, Wd, y, T, ws=None, stream=None):
    """upipe_mlp_fwd: x [L, D], Wgu [2F, D] (gate rows, then up rows),
    Wd [D, F], y [L, D] (written), all bf16; T rows per tile."""
    L, D = x.shape
    F = Wd.shape[1]
    _expect(x, (L, D), torch.bfloat16, "x")
    _expect(Wgu, (2 * F, D), torch.bfloat16, "Wgu")
    _expect(Wd, (D, F), torch.bfloat16, "Wd")
    _expect(y, (L, D), torch.bfloat16, "y")
    _on_device(x=x, Wgu=Wgu, Wd=Wd, y=y)
    ws, nbytes = _tile_ws(mlp_workspace_bytes(L, D, F, T, 0), ws, x.device)
    c = MlpCfg(L, D, F, T)
    _check(lib().upipe_mlp_fwd(ctypes.byref(c), _ptr(x), _ptr(Wgu), _ptr(Wd), _ptr(y), _ptr(ws), nbytes,
                               _stream(stream)), "upipe_mlp_fwd")


def mlp_bwd(x, Wgu, Wd, dy, dx, dWgu, dWd, T, ws=None, stream=None):
    """upipe_mlp_bwd: dy, dx [L, D] bf16; dWgu [2F, D], dWd [D, F] fp32."""
    L, D = x.shape
    F = Wd.shape[1]
    _expect(x, (L, D), torch.bfloat16, "x")
    _expect(Wgu, (2 * F, D), torch.bfloat16, "Wgu")
    _expect(Wd, (D, F), torch.bfloat16, "Wd")
    _expect(dy, (L, D), torch.bfloat16, "dy")
    _expect(dx, (L, D), torch.bfloat16, "dx")
    _expect(dWgu, (2 * F, D), torch.float32, "dWgu")
    _expect(dWd, (D, F), torch.float32, "dWd")
    _on_device(x=x, Wgu=Wgu, Wd=Wd, dy=dy, dx=dx, dWgu=dWgu, dWd=dWd)
    ws, nbytes = _tile_ws(mlp_workspace_bytes(L, D, F, T, 1), ws, x.device)
    c = MlpCfg(L, D, F, T)
    _check(lib().upipe_mlp_bwd(ctypes.byref(c), _ptr(x), _ptr(Wgu), _ptr(Wd), _ptr(dy), _ptr(dx), _ptr(dWgu),
                               _ptr(dWd), _ptr(ws), nbytes, _stream(stream)), "upipe_mlp_bwd")


def ce_fwd_bwd(h, W, labels, scale, loss, dh, dW, T, ws=None, stream=None):
    """upipe_ce_fwd_bwd: h [L, D] bf16, W [V, D] bf16, labels [L] int32,
    loss [L] fp32, dh [L, D] bf16, dW [V, D] fp32 (written)."""
    L, D = h.shape
    V = W.shape[0]
    _expect(h, (L, D), torch.bfloat16, "h")
    _expect(W, (V, D), torch.bfloat16, "W")
    _expect(labels, (L,), torch.int32, "labels")
    _expect(loss, (L,), torch.float32, "loss")
    _expect(dh, (L, D), torch.bfloat16, "dh")
    _expect(dW, (V, D), torch.float32, "dW")
    _on_device(h=h, W=W, labels=labels, loss=loss, dh=dh, dW=dW)
    ws, nbytes = _tile_ws(ce_workspace_bytes(L, D, V, T), ws, h.device)
    c = CeCfg(L, D, V, T)
    _check(lib().upipe_ce_fwd_bwd(ctypes.byref(c), _ptr(h), _ptr(W), _ptr(labels), float(scale), _ptr(loss),
                                  _ptr(dh), _ptr(dW), _ptr(ws), nbytes, _stream(stream)), "upipe_ce_fwd_bwd")


def mlp_forward(x, Wgu, Wd, T):
    y = torch.empty_like(x)
    mlp_fwd(x, Wgu, Wd, y, T)
    return y


def mlp_backward(x, Wgu, Wd, dy, T):
    dx = torch.empty_like(x)
    dWgu = torch.empty(Wgu.shape, dtype=torch.float32, device=x.device)
    dWd = torch.empty(Wd.shape, dtype=torch.float32, device=x.device)
    mlp_bwd(x, Wgu, Wd, dy, dx, dWgu, dWd, T)
    return dx, dWgu, dWd


def ce_loss(h, W, labels, scale, T):
    """Returns (loss [L] fp32, dh [L, D] bf16, dW [V, D] fp32)."""
    loss = torch.empty(h.shape[0], dtype=torch.float32, device=h.device)
    dh = torch.empty_like(h)
    dW = torch.empty(W.shape, dtype=torch.float32, device=h.device)
    ce_fwd_bwd(h, W, labels, scale, loss, dh, dW, T)
    return loss, dh, dW
