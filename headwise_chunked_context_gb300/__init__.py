"""Head-chunked GQA/RoPE causal attention layer for GB300 (sm_103a), with the
sequence-tiled MLP and loss of the same block.

The compute path is the C-ABI library ``libupipe.so`` built from ``csrc/``;
``headwise_chunked_context_gb300.upipe`` is its thin ctypes binding,
``modules`` its autograd front end and ``untied_ulysses`` the chunk loop
across ranks.  Importing this package loads nothing: the library is opened
on first use and a missing library is an error, never a fallback.
"""

__all__ = ["upipe", "synth", "modules", "untied_ulysses"]
