"""GB300-native gated delta rule (Gated DeltaNet recurrence).

The compute path is the C-ABI library `libgdr.so` (hand-written sm_103a CUDA,
declared in include/gdr.h). This package is a thin binding over it:

    from gated_delta_rule_03_gb300 import chunk_fwd, decode_step

Importing the package loads nothing; the first call loads the library and
raises if it is missing. There is no CPU fallback. The submodule `inputs`
(seeded synthetic inputs) can be imported on its own.
"""
_OPS = ("GdrError", "chunk_fwd", "chunk_fwd_workspace_size", "decode_step", "library_path",
        "read_device_status", "status_string")

__all__ = list(_OPS)


def __getattr__(name):
    if name in _OPS:
        from . import ops
        return getattr(ops, name)
    raise AttributeError(name)
