"""Static rules of the CUDA sources (CPU): every barrier wait goes through the
bounded helpers of sm103_ptx.cuh, those helpers take a limit, and no kernel
traps or asserts on the device."""

import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "headwise_chunked_context_gb300",
                    "csrc")
HELPERS = os.path.join(CSRC, "sm103_ptx.cuh")


def _sources():
    return {f: open(os.path.join(CSRC, f)).read() for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh"))}


def test_kernels_wait_only_through_the_helpers():
    for name, text in _sources().items():
        if name == "sm103_ptx.cuh":
            continue
        assert "mbarrier.try_wait" not in text and "mbarrier.test_wait" not in text, name


def test_looping_helpers_are_bounded():
    text = open(HELPERS).read()
    # Every helper that loops on a barrier takes the wait control (abort flag,
    # status word, limit) or, while unwinding, the status word.
    for fn in ("mbar_wait", "mbar_spin", "warp_wait"):
        sig = re.search(r"\b" + fn + r"\(([^)]*)\)\s*\{", text)
        assert sig and "const WaitCtl&" in sig.group(1), fn
    sig = re.search(r"\bmbar_wait_drain\(([^)]*)\)\s*\{", text)
    assert sig and "int* status" in sig.group(1)
    # The loops in those helpers compare a clock against a limit.
    for fn in ("mbar_wait", "mbar_spin", "mbar_wait_drain", "warp_wait"):
        body = text[re.search(r"\b" + fn + r"\(", text).start():]
        body = body[:body.index("\n}\n")]
        assert "sm_cycles()" in body, fn


def test_no_device_trap_or_assert():
    for name, text in _sources().items():
        code = re.sub(r"//[^\n]*", "", text)
        assert "__trap" not in code, name
        assert re.search(r"(?<!static_)\bassert\s*\(", code) is None, name
