"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the attention layer: it only draws
random tensors.  Values are drawn in fp32 from a seeded ``torch.Generator``
and rounded once to bf16; the oracle receives the same bf16 values (upcast
to fp64), the CUDA path receives them as bf16.

Seeds: x=0, Wqkv=1, Wo=2, dout=3 (layer inputs); q=0, k=1, v=2, dO=3 (core
inputs); 10..13 (MLP inputs), 20..22 (loss inputs).  Distributions: activations and upstream gradients ~ N(0, 1),
weights ~ N(0, 0.02).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class LayerShape:
    L: int
    D: int
    H: int
    Hkv: int
    d: int = 128
    U: int = 0
    theta: float = 500000.0

    @property
    def qkv_rows(self) -> int:
        return (self.H + 2 * self.Hkv) * self.d


def _randn(shape, seed, std=1.0, device="cpu", chunk_rows=1 << 16):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    # Draw row blocks in fp32 and round each to bf16, so that large inputs
    # never need a full fp32 copy.
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        blk = torch.randn((r1 - r0, flat.shape[1]), generator=g, dtype=torch.float32, device=device)
        if std != 1.0:
            blk.mul_(std)
        flat[r0:r1].copy_(blk)
    return out


def layer_inputs(s: LayerShape, device="cpu", w_std=0.02):
    """x [L, D], Wqkv [(H+2Hkv) d, D], Wo [D, H d], dout [L, D], all bf16."""
    x = _randn((s.L, s.D), 0, 1.0, device)
    wqkv = _randn((s.qkv_rows, s.D), 1, w_std, device)
    wo = _randn((s.D, s.H * s.d), 2, w_std, device)
    dout = _randn((s.L, s.D), 3, 1.0, device)
    return x, wqkv, wo, dout


def core_inputs(L: int, H: int, Hkv: int, d: int = 128, device="cpu"):
    """q [L, H, d], k, v [L, Hkv, d], dO [L, H, d], all bf16 ~ N(0, 1)."""
    q = _randn((L, H, d), 0, 1.0, device)
    k = _randn((L, Hkv, d), 1, 1.0, device)
    v = _randn((L, Hkv, d), 2, 1.0, device)
    do = _randn((L, H, d), 3, 1.0, device)
    return q, k, v, do


def mlp_inputs(L: int, D: int, F: int, device="cpu", w_std=0.02):
    """x [L, D], Wgu [2F, D] (gate rows, then up rows), Wd [D, F], dy [L, D],
    all bf16 (seeds 10..13)."""
    x = _randn((L, D), 10, 1.0, device)
    wgu = _randn((2 * F, D), 11, w_std, device)
    wd = _randn((D, F), 12, w_std, device)
    dy = _randn((L, D), 13, 1.0, device)
    return x, wgu, wd, dy


def ce_inputs(L: int, D: int, V: int, device="cpu", w_std=0.02, ignore_every=17):
    """h [L, D], W [V, D] bf16 (seeds 20, 21) and int32 labels [L] uniform
    over the vocabulary (seed 22), every `ignore_every`-th one set to -100
    (ignored)."""
    h = _randn((L, D), 20, 1.0, device)
    w = _randn((V, D), 21, w_std, device)
    g = torch.Generator(device="cpu")
    g.manual_seed(22)
    labels = torch.randint(0, V, (L,), generator=g, dtype=torch.int32)
    if ignore_every:
        labels[ignore_every - 1::ignore_every] = -100
    return h, w, labels.to(device)


# The five workloads, by name.
TINY = LayerShape(L=1024, D=1024, H=8, Hkv=2, d=128, U=2)
LLAMA8B = LayerShape(L=32768, D=4096, H=32, Hkv=8, d=128, U=8)
SLICE_1M = dict(L=1048576, H=4, Hkv=1, d=128, U=1)
QWEN32B = LayerShape(L=131072, D=5120, H=64, Hkv=8, d=128, U=8)
LONG_SWEEP_L = (65536, 262144, 1048576, 2097152)
LONG_SWEEP = LayerShape(L=65536, D=4096, H=32, Hkv=8, d=128, U=4)
