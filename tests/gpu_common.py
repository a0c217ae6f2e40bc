"""Shared setup of the GPU parity tests: builds the library if needed and
moves seeded CPU inputs to cuda:0."""

import os

import numpy as np
import torch

from headwise_chunked_context_gb300 import upipe


def ensure_lib():
    if not os.path.exists(upipe.LIB_PATH):
        from headwise_chunked_context_gb300 import build
        build.build()
    return upipe.lib()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def dev(*ts):
    return [t.to("cuda:0") for t in ts]


def status_ok():
    code = upipe.last_device_status()
    assert code == 0, f"device status {code}: {upipe.strerror(code)}"
