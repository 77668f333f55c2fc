"""Thin ctypes binding over libgdr.so (include/gdr.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. PyTorch provides device memory and the current stream. If the
library is missing the first call raises GdrError; nothing falls back to the CPU.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgdr.so")
_lib = None

GDR_F32, GDR_BF16 = 0, 1
_DTYPES = {torch.float32: GDR_F32, torch.bfloat16: GDR_BF16}
# the recurrence's write rule (gdr_options.rule)
RULES = {"delta": 0, "additive": 1}
# the forget gate's granularity (gdr_options.decay): one rate per head, or per key channel
DECAYS = {"head": 0, "channel": 1}


class GdrOptions(ctypes.Structure):
    """struct gdr_options of gdr.h."""
    _fields_ = [("rule", ctypes.c_int), ("out_norm_eps", ctypes.c_float),
                ("out_gate", ctypes.c_void_p), ("out_norm_weight", ctypes.c_void_p),
                ("prologue", ctypes.c_int), ("decay", ctypes.c_int),
                ("gate_A", ctypes.c_void_p)]


def _options(rule, out_gate=None, out_norm_weight=None, out_norm_eps=0.0, prologue=False,
             gate_A=None, decay="head"):
    if rule not in RULES:
        raise ValueError(f"unknown rule {rule!r}; expected one of {sorted(RULES)}")
    opt = GdrOptions(RULES[rule], float(out_norm_eps) if out_gate is not None else 0.0,
                     None if out_gate is None else out_gate.data_ptr(),
                     None if out_norm_weight is None else out_norm_weight.data_ptr(),
                     1 if prologue else 0, DECAYS[decay],
                     None if gate_A is None else gate_A.data_ptr())
    return ctypes.byref(opt)


def _decay_of(log_alpha, lead, dk):
    """'head' for log_alpha of shape `lead`, 'channel' for `lead` + (dk,)."""
    shape = tuple(log_alpha.shape)
    if shape == tuple(lead):
        return "head"
    if shape == tuple(lead) + (dk,):
        return "channel"
    raise ValueError(f"log_alpha must have shape {tuple(lead)} (one rate per head) or "
                     f"{tuple(lead) + (dk,)} (one rate per key channel), got {shape}")


def _check_prologue(prologue, gate_A, H, device):
    if gate_A is None:
        return
    if not prologue:
        raise ValueError("gate_A needs prologue=True")
    _need(gate_A, "gate_A", torch.float32, device)
    if gate_A.numel() != H:
        raise ValueError(f"gate_A must have {H} entries")


def _check_out_step(out_gate, out_norm_weight, like, dv):
    if out_gate is None:
        if out_norm_weight is not None:
            raise ValueError("out_norm_weight needs out_gate")
        return
    _need(out_gate, "out_gate", like.dtype, like.device)
    if tuple(out_gate.shape) != tuple(like.shape):
        raise ValueError(f"out_gate must have shape {tuple(like.shape)}")
    if out_norm_weight is not None:
        _need(out_norm_weight, "out_norm_weight", torch.float32, like.device)
        if out_norm_weight.numel() != dv:
            raise ValueError(f"out_norm_weight must have {dv} entries")


class GdrError(RuntimeError):
    """A libgdr call returned a negative status."""

    def __init__(self, status, what, detail=None):
        # detail: the status text; read from the library unless given (it is given when
        # the library itself cannot be loaded)
        self.status = status
        if detail is None:
            detail = status_string(status)
        super().__init__(f"{what}: {detail} ({status})")


def library_path():
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise GdrError(-5, f"libgdr.so not found at {_LIB_PATH}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`",
                       detail="the CUDA library is not built")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, fp, i64, c_int = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.gdr_status_string.argtypes = [c_int]
    lib.gdr_status_string.restype = ctypes.c_char_p
    lib.gdr_chunk_fwd_workspace_size.argtypes = [i64, i64, c_int, c_int, c_int, c_int, c_int]
    lib.gdr_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    lib.gdr_chunk_fwd_workspace_size_ex.argtypes = [i64, i64, c_int, c_int, c_int, c_int, c_int,
                                                    ctypes.c_void_p]
    lib.gdr_chunk_fwd_workspace_size_ex.restype = ctypes.c_size_t
    lib.gdr_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, fp, vp, i64, i64, c_int, c_int, c_int,
                                  c_int, c_int, vp, fp, vp, ctypes.c_size_t, vp]
    lib.gdr_chunk_fwd.restype = c_int
    lib.gdr_chunk_fwd_ex.argtypes = [vp, vp, vp, fp, fp, fp, vp, i64, i64, c_int, c_int, c_int,
                                     c_int, c_int, vp, fp, vp, ctypes.c_size_t, vp, vp]
    lib.gdr_chunk_fwd_ex.restype = c_int
    lib.gdr_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, i64, c_int, c_int, c_int, c_int,
                                    vp]
    lib.gdr_decode_step.restype = c_int
    lib.gdr_decode_step_ex.argtypes = [vp, vp, vp, fp, fp, fp, vp, i64, c_int, c_int, c_int, c_int,
                                       vp, vp]
    lib.gdr_decode_step_ex.restype = c_int
    lib.gdr_chunk_fwd_path.argtypes = [c_int, c_int, c_int]
    lib.gdr_chunk_fwd_path.restype = c_int
    lib.gdr_chunk_fwd_path_ex.argtypes = [c_int, c_int, c_int, vp]
    lib.gdr_chunk_fwd_path_ex.restype = c_int
    lib.gdr_chunk_fwd_kernel_launches.argtypes = [i64, i64, c_int, c_int, c_int, c_int, c_int,
                                                  c_int]
    lib.gdr_chunk_fwd_kernel_launches.restype = c_int
    lib.gdr_chunk_fwd_schedule.argtypes = [i64, i64, c_int, c_int, c_int, c_int, c_int, c_int]
    lib.gdr_chunk_fwd_schedule.restype = c_int
    lib.gdr_chunk_fwd_schedule_model.argtypes = [i64, i64, c_int, c_int, c_int, c_int, c_int, c_int,
                                                 c_int, c_int]
    lib.gdr_chunk_fwd_schedule_model.restype = c_int
    lib.gdr_read_device_status.argtypes = [vp, ctypes.POINTER(c_int), vp]
    lib.gdr_read_device_status.restype = c_int
    _lib = lib
    return lib


def status_string(status):
    return _load().gdr_status_string(int(status)).decode()


def _check(status, what):
    if status != 0:
        raise GdrError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def chunk_fwd_workspace_size(num_seqs, total_tokens, H, dk, dv, chunk=64, dtype=torch.bfloat16,
                             decay="head", prologue=False):
    """Workspace bytes gdr_chunk_fwd needs (0 if the sizes are unsupported); decay
    "channel" (per-channel rates, whose path also depends on the prologue) through
    gdr_chunk_fwd_workspace_size_ex."""
    lib = _load()
    if decay == "head":
        return int(lib.gdr_chunk_fwd_workspace_size(int(num_seqs), int(total_tokens), int(H),
                                                    int(dk), int(dv), int(chunk), _DTYPES[dtype]))
    opt = GdrOptions(0, 0.0, None, None, int(bool(prologue)), DECAYS[decay], None)
    return int(lib.gdr_chunk_fwd_workspace_size_ex(int(num_seqs), int(total_tokens), int(H),
                                                   int(dk), int(dv), int(chunk), _DTYPES[dtype],
                                                   ctypes.addressof(opt)))


def chunk_fwd(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, num_seqs=None, chunk=64,
              o=None, S_final=None, workspace=None, stream=None, rule="delta", out_gate=None,
              out_norm_weight=None, out_norm_eps=1e-6, prologue=False, gate_A=None):
    """Chunked prefill (gdr_chunk_fwd).

    q, k [T, H, dk]; v [T, H, dv] (fp32 or bf16); beta [T, H] fp32; log_alpha [T, H]
    fp32 (one rate per head), or [T, H, dk] (one rate per key channel, gdr_options.decay
    GDR_DECAY_CHANNEL: tensor cores for bf16 with dk = dv = 128, else the exact fp32
    path);
    S0 [num_seqs, H, dk, dv] fp32 or None; cu_seqlens [num_seqs+1] int32 or None
    (then `num_seqs` equal sequences, default 1). Optional preallocated o,
    S_final and workspace (uint8) tensors are used as given. rule: "delta" (the gated
    delta rule) or "additive" (S <- alpha S + beta k v^T). out_gate [T, H, dv] (o's
    dtype): apply the layer's output step o <- o / rms(o) * out_norm_weight * silu(out_gate)
    over each head's dv entries. prologue=True: q and k are raw (scaled to unit length in
    the kernels) and log_alpha, beta hold the gate pre-activations a, b (log alpha =
    -gate_A[h] softplus(a), beta = sigmoid(b)); see gdr_options in gdr.h. Returns
    (o, S_final).
    """
    lib = _load()
    _need(q, "q")
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported dtype {dt}")
    T, H, dk = q.shape
    dv = v.shape[-1]
    _need(k, "k", dt, dev)
    _need(v, "v", dt, dev)
    _need(log_alpha, "log_alpha", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    decay = _decay_of(log_alpha, (T, H), dk)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
        n = cu_seqlens.numel() - 1
    else:
        n = 1 if num_seqs is None else int(num_seqs)
    if S0 is not None:
        _need(S0, "S0", torch.float32, dev)
    if o is None:
        o = torch.empty((T, H, dv), dtype=dt, device=dev)
    if S_final is None:
        S_final = torch.empty((n, H, dk, dv), dtype=torch.float32, device=dev)
    _need(o, "o", dt, dev)
    _need(S_final, "S_final", torch.float32, dev)
    _check_out_step(out_gate, out_norm_weight, o, dv)
    _check_prologue(prologue, gate_A, H, dev)
    ws_bytes = chunk_fwd_workspace_size(n, T, H, dk, dv, chunk, dt, decay, prologue)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", device=dev)
    st = lib.gdr_chunk_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
                              _ptr(cu_seqlens), n, T, H, dk, dv, int(chunk), _DTYPES[dt], _ptr(o),
                              _ptr(S_final), _ptr(workspace),
                              workspace.numel() * workspace.element_size(),
                              _options(rule, out_gate, out_norm_weight, out_norm_eps, prologue,
                                       gate_A, decay),
                              _stream_handle(stream, dev))
    _check(st, "gdr_chunk_fwd_ex")
    return o, S_final


def read_device_status(workspace, stream=None):
    """Status word the last gdr_chunk_fwd left in `workspace` (synchronises the stream)."""
    out = ctypes.c_int(0)
    st = _load().gdr_read_device_status(_ptr(workspace), ctypes.byref(out),
                                        _stream_handle(stream, workspace.device))
    _check(st, "gdr_read_device_status")
    return out.value


def decode_step(q, k, v, log_alpha, beta, S, o=None, stream=None, rule="delta", out_gate=None,
                out_norm_weight=None, out_norm_eps=1e-6, prologue=False, gate_A=None):
    """One decode step (gdr_decode_step_ex): q, k [N, H, dk]; v [N, H, dv];
    beta [N, H] fp32; log_alpha [N, H] fp32, or [N, H, dk] (one rate per key channel);
    S [N, H, dk, dv] fp32 updated in place; rule "delta" (the gated delta rule) or
    "additive" (S <- alpha S + beta k v^T). Returns o [N, H, dv]."""
    lib = _load()
    _need(q, "q")
    dev, dt = q.device, q.dtype
    N, H, dk = q.shape
    dv = v.shape[-1]
    _need(k, "k", dt, dev)
    _need(v, "v", dt, dev)
    _need(log_alpha, "log_alpha", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(S, "S", torch.float32, dev)
    decay = _decay_of(log_alpha, (N, H), dk)
    if o is None:
        o = torch.empty((N, H, dv), dtype=dt, device=dev)
    _need(o, "o", dt, dev)
    _check_out_step(out_gate, out_norm_weight, o, dv)
    _check_prologue(prologue, gate_A, H, dev)
    st = lib.gdr_decode_step_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S),
                                _ptr(o), N, H, dk, dv, _DTYPES[dt],
                                _options(rule, out_gate, out_norm_weight, out_norm_eps, prologue,
                                         gate_A, decay),
                                _stream_handle(stream, dev))
    _check(st, "gdr_decode_step_ex")
    return o


# The dominant kernel and the product arithmetic of each kernel path (see
# gdr_chunk_fwd_path in gdr.h).
_PATHS = {
    0: dict(main_kernel="exact_chain_kernel", compute_dtype="f32"),
    1: dict(main_kernel="tc_chain_kernel", compute_dtype="bf16"),
    2: dict(main_kernel="channel_prep_kernel", compute_dtype="bf16"),
}
PATH_CHANNEL_TENSOR = 2  # GDR_PATH_CHANNEL_TENSOR


def chunk_fwd_path(dk, dv, dtype, decay="head", prologue=False):
    """0 (exact fp32 path), 1 (tensor cores, one rate per head) or 2 (tensor cores,
    one rate per key channel), from gdr_chunk_fwd_path_ex."""
    opt = GdrOptions(0, 0.0, None, None, int(bool(prologue)), DECAYS[decay], None)
    st = _load().gdr_chunk_fwd_path_ex(int(dk), int(dv), _DTYPES[dtype], ctypes.addressof(opt))
    if st < 0:
        raise GdrError(st, "gdr_chunk_fwd_path_ex")
    return st


def chunk_fwd_kernel_launches(num_seqs, total_tokens, H, dk, dv, dtype, varlen=False,
                              decay="head"):
    """Kernels one gdr_chunk_fwd call launches for these sizes on the current device
    (varlen: the call passes cu_seqlens)."""
    if decay == "channel":  # either per-channel path: plan, per-chunk operands, chain
        chunk_fwd_path(dk, dv, dtype, decay)
        return 3 if total_tokens > 0 else 1
    st = _load().gdr_chunk_fwd_kernel_launches(int(num_seqs), int(total_tokens), int(H), int(dk),
                                               int(dv), 64, _DTYPES[dtype], int(bool(varlen)))
    if st < 0:
        raise GdrError(st, "gdr_chunk_fwd_kernel_launches")
    return st


SCHEDULE_SEGMENTED = 16  # GDR_SCHEDULE_SEGMENTED


def chunk_fwd_schedule(num_seqs, total_tokens, H, dk, dv, dtype, varlen=False, decay="head"):
    """Schedule of a gdr_chunk_fwd call with these sizes on the current device: 0 for the
    fused tensor-core schedule, 1 .. 8 phases of the phased one, or SCHEDULE_SEGMENTED + n
    for the segmented one with n segments per sequence (the exact path: one phase)."""
    if decay == "channel":
        return 1
    st = _load().gdr_chunk_fwd_schedule(int(num_seqs), int(total_tokens), int(H), int(dk),
                                        int(dv), 64, _DTYPES[dtype], int(bool(varlen)))
    if st < 0:
        raise GdrError(st, "gdr_chunk_fwd_schedule")
    return st


def chunk_fwd_schedule_model(num_seqs, total_tokens, H, dk, dv, dtype, sms, varlen=False,
                             cooperative=True):
    """The schedule a device with `sms` SMs would take for these sizes (no CUDA call)."""
    st = _load().gdr_chunk_fwd_schedule_model(int(num_seqs), int(total_tokens), int(H), int(dk),
                                              int(dv), 64, _DTYPES[dtype], int(bool(varlen)),
                                              int(sms), int(bool(cooperative)))
    if st < 0:
        raise GdrError(st, "gdr_chunk_fwd_schedule_model")
    return st


def chunk_fwd_main_kernel(dk, dv, dtype, schedule=None, decay="head"):
    """Name of the kernel that dominates a gdr_chunk_fwd call for these sizes. The fused
    schedule (0) of the tensor-core path runs the solve and the chains in one kernel; the
    other paths are dominated by their chain."""
    path = chunk_fwd_path(dk, dv, dtype, decay)
    if path == 1 and schedule == 0:
        return "tc_fused_kernel"
    return _PATHS[path]["main_kernel"]


def chunk_fwd_compute_dtype(dk, dv, dtype, decay="head"):
    """Arithmetic type of the products on the path taken (f32 SIMT or bf16 tensor cores)."""
    return _PATHS[chunk_fwd_path(dk, dv, dtype, decay)]["compute_dtype"]
