"""Head-chunked GQA/RoPE causal attention layer for GB300 (sm_103a).

The compute path is the C-ABI library ``libupipe.so`` built from ``csrc/``;
``headwise_chunked_context_gb300.upipe`` is its thin ctypes binding.  Importing
this package loads nothing: the library is opened on first use and a missing
library is an error, never a fallback.
"""

__all__ = ["upipe", "synth"]
