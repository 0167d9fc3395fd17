"""GB300-native causal linear self-attention in SLiM's chunked, sub-linear-memory form.

The compute path is the C-ABI library ``libslim_attn.so`` (hand-written sm_103a
CUDA kernels, see ``csrc/``); ``binding`` marshals torch tensors into it.  The
binding is imported lazily so that ``inputs`` (the seeded workloads) can be
used without loading the library.
"""
import importlib

__all__ = ["slim_attn_fwd", "slim_attn_bwd", "binding", "inputs"]


def __getattr__(name):
    if name in ("binding", "inputs"):
        return importlib.import_module("." + name, __name__)
    if name in ("slim_attn_fwd", "slim_attn_bwd", "SlimError", "library_path"):
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
