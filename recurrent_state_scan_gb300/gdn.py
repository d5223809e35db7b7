"""Thin Python binding of libgdn's C ABI (argument marshalling only).

Every step of the scan runs in libgdn's CUDA kernels; PyTorch only supplies
device memory and the stream.  The entry points keep the C names:
``gdn_prefill``, ``gdn_decode_step``, ``gdn_prefill_workspace_bytes``,
``gdn_last_device_status``, ``gdn_status_string``.  If the library cannot be
loaded every call raises -- there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED = 0, 1, 2
GDN_ERR_CUDA, GDN_ERR_DEVICE_CHECK, GDN_ERR_TIMEOUT = 3, 4, 5
GDN_F32, GDN_BF16, GDN_F16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: GDN_F32, torch.bfloat16: GDN_BF16, torch.float16: GDN_F16}

# Every symbol include/gdn.h declares.
EXPORTS = ("gdn_prefill_workspace_bytes", "gdn_prefill", "gdn_decode_step",
           "gdn_prefill_plan", "gdn_last_device_status", "gdn_status_string",
           "gdn_last_error_message", "gdn_prefill_noalloc", "gdn_decode_step_slots",
           "gdn_scan_window", "gdn_scan_variant", "gdn_causal_conv", "gdn_causal_conv_slots",
           "gdn_gated_rmsnorm", "gdn_set_wait_budget", "gdn_decode_layer", "gdn_prefill_variant",
           "gdn_prefill_norm", "gdn_prefill_variant_workspace_bytes", "gdn_prefill_variant_plan",
           "gdn_prefill_layer", "gdn_prefill_layer_workspace_bytes")
PATH_SIMT, PATH_TC, PATH_TC_TP = 1, 2, 3
# gdn_rule codes.
RULES = {"gated_delta": 0, "delta": 1, "gated": 2, "linear": 3}
# gdn_activation codes.
ACTIVATIONS = {"none": 0, "silu": 1, "swish": 1, "sigmoid": 2}


class GdnShape(ctypes.Structure):
    _fields_ = [("io_dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("seqlen", ctypes.c_int64), ("num_seqs", ctypes.c_int32),
                ("h_qk", ctypes.c_int32), ("h_v", ctypes.c_int32),
                ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32)]


class GdnVariant(ctypes.Structure):
    _fields_ = [("rule", ctypes.c_int32), ("decay_per_key", ctypes.c_int32),
                ("beta_shared", ctypes.c_int32)]


class GdnConvShape(ctypes.Structure):
    _fields_ = [("io_dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("seqlen", ctypes.c_int64), ("channels", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("dilation", ctypes.c_int32),
                ("channels_last", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("state_window", ctypes.c_int32)]


class GdnLayerParams(ctypes.Structure):
    _fields_ = [("conv_kernel", ctypes.c_int32), ("conv_activation", ctypes.c_int32),
                ("norm_activation", ctypes.c_int32), ("norm_epsilon", ctypes.c_float)]


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_name(status)}: {message}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdn.so (building it first if allowed).  Raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB) or (build_if_missing and not _build.up_to_date()):
        if not build_if_missing:
            raise GdnError(GDN_ERR_CUDA, f"libgdn is not built ({_build.LIB})")
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    P = ctypes.c_void_p
    S = ctypes.POINTER(GdnShape)
    lib.gdn_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_prefill_workspace_bytes.argtypes = [S]
    lib.gdn_prefill.restype = ctypes.c_int
    lib.gdn_prefill.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P,
                                ctypes.c_size_t, P]
    lib.gdn_scan_window.restype = ctypes.c_int
    lib.gdn_scan_window.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_float, P, P,
                                    ctypes.c_int32, P]
    CS = ctypes.POINTER(GdnConvShape)
    lib.gdn_causal_conv.restype = ctypes.c_int
    lib.gdn_causal_conv.argtypes = [CS, P, P, P, P, P, P, P]
    lib.gdn_causal_conv_slots.restype = ctypes.c_int
    lib.gdn_causal_conv_slots.argtypes = [CS, P, P, P, P, ctypes.c_int64, P, P, P]
    lib.gdn_gated_rmsnorm.restype = ctypes.c_int
    lib.gdn_gated_rmsnorm.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, P, P, P,
                                      ctypes.c_float, ctypes.c_int32, P, P]
    lib.gdn_scan_variant.restype = ctypes.c_int
    lib.gdn_scan_variant.argtypes = [S, ctypes.POINTER(GdnVariant), P, P, P, P, P, P, P, P, P,
                                     ctypes.c_float, P, P, P]
    lib.gdn_decode_step_slots.restype = ctypes.c_int
    lib.gdn_decode_step_slots.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_int64, P,
                                          ctypes.c_float, P, P]
    lib.gdn_prefill_noalloc.restype = ctypes.c_int
    lib.gdn_prefill_noalloc.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P]
    lib.gdn_decode_step.restype = ctypes.c_int
    lib.gdn_decode_step.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_float, P, P]
    lib.gdn_prefill_plan.restype = ctypes.c_int
    lib.gdn_prefill_plan.argtypes = [S, ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int32)]
    lib.gdn_last_device_status.restype = ctypes.c_int
    lib.gdn_last_device_status.argtypes = [P]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_last_error_message.restype = ctypes.c_char_p
    lib.gdn_last_error_message.argtypes = []
    lib.gdn_set_wait_budget.restype = ctypes.c_int
    lib.gdn_set_wait_budget.argtypes = [ctypes.c_int64]
    lib.gdn_prefill_variant.restype = ctypes.c_int
    lib.gdn_prefill_variant.argtypes = [S, ctypes.POINTER(GdnVariant), P, P, P, P, P, P, P, P, P,
                                        ctypes.c_float, P, P, P, ctypes.c_size_t, P]
    lib.gdn_prefill_variant_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_prefill_variant_workspace_bytes.argtypes = [S, ctypes.POINTER(GdnVariant)]
    lib.gdn_prefill_variant_plan.restype = ctypes.c_int
    lib.gdn_prefill_variant_plan.argtypes = [S, ctypes.POINTER(GdnVariant), ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int32)]
    lib.gdn_prefill_norm.restype = ctypes.c_int
    lib.gdn_prefill_norm.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_float, P, P,
                                     ctypes.c_float, ctypes.c_int32, ctypes.c_int32, P, P, P,
                                     ctypes.c_size_t, P]
    lib.gdn_decode_layer.restype = ctypes.c_int
    lib.gdn_decode_layer.argtypes = [S, ctypes.POINTER(GdnLayerParams), P, P, P, P, P, P, P, P, P,
                                     P, ctypes.c_float, P, P, P, P]
    lib.gdn_prefill_layer.restype = ctypes.c_int
    lib.gdn_prefill_layer.argtypes = [S, ctypes.POINTER(GdnLayerParams), P, P, P, P, P, P, P, P, P, P, P,
                                      ctypes.c_float, P, P, P, P, ctypes.c_int32, P, ctypes.c_size_t, P]
    lib.gdn_prefill_layer_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_prefill_layer_workspace_bytes.argtypes = [S]
    _lib = lib
    return lib


def status_name(status: int) -> str:
    try:
        return load().gdn_status_string(int(status)).decode()
    except Exception:  # the name is only cosmetic
        return f"status {status}"


def _check(status: int):
    if status != GDN_OK:
        raise GdnError(status, load().gdn_last_error_message().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise GdnError(GDN_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")


def make_shape(io_dtype: int, batch: int, seqlen: int, num_seqs: int, h_qk: int, h_v: int,
               d_k: int, d_v: int) -> GdnShape:
    return GdnShape(io_dtype, batch, seqlen, num_seqs, h_qk, h_v, d_k, d_v)


def _shape_of(q, v, cu_seqlens) -> GdnShape:
    if q.dim() != 4 or v.dim() != 4:
        raise GdnError(GDN_ERR_INVALID_ARG, "q and v must be [B, T, H, D]")
    B, T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[2], v.shape[3]
    if q.dtype not in _DTYPE_CODE:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unsupported io dtype {q.dtype}")
    n = B if cu_seqlens is None else cu_seqlens.numel() - 1
    return make_shape(_DTYPE_CODE[q.dtype], B, T, n, h_qk, h_v, d_k, d_v)


def gdn_prefill_workspace_bytes(shape: GdnShape) -> int:
    return int(load().gdn_prefill_workspace_bytes(ctypes.byref(shape)))


def gdn_prefill(q, k, v, a, b, A_log, dt_bias, state_in=None, cu_seqlens=None,
                scale: float = 0.0, *, o=None, state_out=None, workspace=None, stream=None):
    """Run the gated delta rule over whole sequences; returns (o, state_out).

    q, k [B,T,h_qk,d_k]; v [B,T,h_v,d_v]; a, b [B,T,h_v] (all one io dtype);
    A_log, dt_bias [h_v] fp32; state_in [N,h_v,d_k,d_v] fp32 or None;
    cu_seqlens int32 [N+1] on the device (then B must be 1) or None.
    """
    lib = load()
    shape = _shape_of(q, v, cu_seqlens)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    if tuple(k.shape) != tuple(q.shape) or tuple(a.shape) != tuple(v.shape[:3]) or \
            tuple(b.shape) != tuple(a.shape):
        raise GdnError(GDN_ERR_INVALID_ARG, "k must match q, and a, b must be [B, T, h_v]")
    if tuple(A_log.shape) != (shape.h_v,) or tuple(dt_bias.shape) != (shape.h_v,):
        raise GdnError(GDN_ERR_INVALID_ARG, "A_log and dt_bias must be [h_v]")
    st_shape = (shape.num_seqs, shape.h_v, shape.d_k, shape.d_v)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
        if tuple(state_in.shape) != st_shape:
            raise GdnError(GDN_ERR_INVALID_ARG, f"state_in must be {st_shape}")
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("o", o, dt)
    if state_out is None:
        state_out = torch.empty(st_shape, dtype=torch.float32, device=v.device)
    else:
        _need_cuda("state_out", state_out, torch.float32)
    need = int(lib.gdn_prefill_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                           _ptr(A_log), _ptr(dt_bias), _ptr(state_in), _ptr(cu_seqlens),
                           float(scale), _ptr(o), _ptr(state_out), _ptr(workspace), ws_bytes,
                           _stream(stream)))
    return o, state_out


# Size of the library's fixed scratch array behind gdn_prefill_noalloc.
PREFILL_NOALLOC_SCRATCH_BYTES = 96 * 1024 * 1024



def gdn_prefill_norm(q, k, v, a, b, A_log, dt_bias, state_in=None, cu_seqlens=None,
                     scale: float = 0.0, *, norm_scale, gate, eps: float = 1e-6,
                     activation: str = "silu", fuse: bool = False, y=None, state_out=None,
                     workspace=None, stream=None):
    """gdn_prefill, then the gated RMS norm of o over each d_v row; returns (y, state_out).

    norm_scale [d_v] and gate (o's shape) in the io dtype; y has o's shape.  fuse: run the
    norm in the tensor-core scan's readout (o never stored) where the path allows; by
    default the norm is a second launch, in place on y."""
    lib = load()
    shape = _shape_of(q, v, cu_seqlens)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("gate", gate),
                    ("norm_scale", norm_scale)):
        _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    if tuple(k.shape) != tuple(q.shape) or tuple(a.shape) != tuple(v.shape[:3]) or \
            tuple(b.shape) != tuple(a.shape):
        raise GdnError(GDN_ERR_INVALID_ARG, "k must match q, and a, b must be [B, T, h_v]")
    if tuple(gate.shape) != tuple(v.shape) or tuple(norm_scale.shape) != (shape.d_v,):
        raise GdnError(GDN_ERR_INVALID_ARG, "gate must match v, norm_scale must be [d_v]")
    if activation not in ("silu", "swish", "sigmoid"):
        raise GdnError(GDN_ERR_INVALID_ARG, "activation is silu or sigmoid")
    st_shape = (shape.num_seqs, shape.h_v, shape.d_k, shape.d_v)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
        if tuple(state_in.shape) != st_shape:
            raise GdnError(GDN_ERR_INVALID_ARG, f"state_in must be {st_shape}")
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    if y is None:
        y = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("y", y, dt)
    if state_out is None:
        state_out = torch.empty(st_shape, dtype=torch.float32, device=v.device)
    else:
        _need_cuda("state_out", state_out, torch.float32)
    need = int(lib.gdn_prefill_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_prefill_norm(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                                _ptr(A_log), _ptr(dt_bias), _ptr(state_in), _ptr(cu_seqlens),
                                float(scale), _ptr(norm_scale), _ptr(gate), float(eps),
                                ACTIVATIONS[activation], int(bool(fuse)), _ptr(y), _ptr(state_out),
                                _ptr(workspace), ws_bytes, _stream(stream)))
    return y, state_out


def gdn_prefill_noalloc(q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, scale: float,
                        *, o, state_out, stream=None):
    """gdn_prefill for callers that may not allocate device memory: the outputs are
    caller-provided and the tensor-core path's scratch is the library's fixed
    96 MiB array, shared by every call on the device (calls that overlap on the GPU
    race on it).  Shapes needing more scratch raise GDN_ERR_INVALID_ARG."""
    lib = load()
    shape = _shape_of(q, v, cu_seqlens)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b), ("o", o)):
        _need_cuda(name, t, dt)
    for name, t in (("A_log", A_log), ("dt_bias", dt_bias), ("state_out", state_out)):
        _need_cuda(name, t, torch.float32)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    st_shape = (shape.num_seqs, shape.h_v, shape.d_k, shape.d_v)
    if tuple(o.shape) != tuple(v.shape) or tuple(state_out.shape) != st_shape:
        raise GdnError(GDN_ERR_INVALID_ARG, f"o must be {tuple(v.shape)} and state_out {st_shape}")
    _check(lib.gdn_prefill_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                   _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(state_in),
                                   _ptr(cu_seqlens), float(scale), _ptr(o), _ptr(state_out),
                                   _stream(stream)))
    return o, state_out


def gdn_decode_step(q, k, v, a, b, A_log, dt_bias, state, scale: float = 0.0, *, o=None,
                    stream=None):
    """One token per sequence; ``state`` [B,h_v,d_k,d_v] fp32 is updated in place.

    q, k [B,1,h_qk,d_k]; v [B,1,h_v,d_v]; a, b [B,1,h_v].  Returns o [B,1,h_v,d_v].
    """
    lib = load()
    shape = _shape_of(q, v, None)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    _need_cuda("state", state, torch.float32)
    if tuple(state.shape) != (shape.batch, shape.h_v, shape.d_k, shape.d_v):
        raise GdnError(GDN_ERR_INVALID_ARG, "state must be [B, h_v, d_k, d_v]")
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("o", o, dt)
    _check(lib.gdn_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                               _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(state), float(scale),
                               _ptr(o), _stream(stream)))
    return o


def gdn_prefill_plan(shape: GdnShape):
    """(path, launches per call) that gdn_prefill takes for ``shape``."""
    path, launches = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().gdn_prefill_plan(ctypes.byref(shape), ctypes.byref(path),
                                   ctypes.byref(launches)))
    return path.value, launches.value


def gdn_prefill_variant_plan(shape: GdnShape, rule: str = "gated_delta", decay_per_key: bool = False,
                             beta_shared: bool = False):
    """(path, launches per call) that gdn_prefill_variant takes for ``shape`` with the
    workspace gdn_prefill_variant_workspace_bytes reports."""
    if rule not in RULES:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unknown rule {rule!r}")
    var = GdnVariant(RULES[rule], int(bool(decay_per_key)), int(bool(beta_shared)))
    path, launches = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load().gdn_prefill_variant_plan(ctypes.byref(shape), ctypes.byref(var), ctypes.byref(path),
                                           ctypes.byref(launches)))
    return path.value, launches.value


def gdn_prefill_layer_workspace_bytes(shape: GdnShape) -> int:
    """The workspace gdn_prefill_layer needs for ``shape`` (0 off the tensor-core shapes)."""
    return int(load().gdn_prefill_layer_workspace_bytes(ctypes.byref(shape)))


def gdn_prefill_variant_workspace_bytes(shape: GdnShape, rule: str = "gated_delta",
                                        decay_per_key: bool = False, beta_shared: bool = False) -> int:
    if rule not in RULES:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unknown rule {rule!r}")
    var = GdnVariant(RULES[rule], int(bool(decay_per_key)), int(bool(beta_shared)))
    return int(load().gdn_prefill_variant_workspace_bytes(ctypes.byref(shape), ctypes.byref(var)))


def shape_of_spec(spec, n_seq: int, total_tokens: int) -> GdnShape:
    io = {"f32": GDN_F32, "bf16": GDN_BF16, "f16": GDN_F16}[spec.io]
    if spec.lengths is not None or spec.varlen_range is not None:
        return make_shape(io, 1, total_tokens, n_seq, spec.h_qk, spec.h_v, spec.d_k, spec.d_v)
    return make_shape(io, spec.batch, spec.seqlen, spec.batch, spec.h_qk, spec.h_v, spec.d_k,
                      spec.d_v)


def _simt_only(spec) -> bool:
    """Specs that run the token-sequential kernel alone: decode and state windows (the
    rules, the shared beta and the per-key-dim decay of a prefill take gdn_prefill's path
    through gdn_prefill_variant)."""
    return bool(spec.decode or getattr(spec, "window", 0))


def gdn_set_wait_budget(cycles: int) -> None:
    """Test hook: cycles a bounded wait of the tensor-core prefill kernels may take before
    the CTA gives up (0: the default, about two seconds)."""
    _check(load().gdn_set_wait_budget(int(cycles)))


def launches_per_call(spec, n_seq: int = 0, total_tokens: int = 0) -> int:
    if _simt_only(spec):
        return 1
    return gdn_prefill_plan(shape_of_spec(spec, n_seq, total_tokens))[1]


def path_dtype(spec, n_seq: int = 0, total_tokens: int = 0) -> str:
    """Arithmetic type of the path: MMA operand type on the tensor-core path, else f32."""
    if _simt_only(spec):
        return "f32"
    path = gdn_prefill_plan(shape_of_spec(spec, n_seq, total_tokens))[0]
    return spec.io if path in (PATH_TC, PATH_TC_TP) else "f32"


def gdn_last_device_status(stream=None) -> int:
    """Synchronise, read and clear the device check word; returns the status code."""
    return int(load().gdn_last_device_status(_stream(stream)))


def gdn_status_string(status: int) -> str:
    return load().gdn_status_string(int(status)).decode()


def gdn_decode_step_slots(q, k, v, a, b, A_log, dt_bias, pool, slots, scale: float = 0.0, *,
                          o=None, stream=None):
    """One token per sequence against a pool of states: sequence b reads and updates
    ``pool[slots[b]]`` in place.  q, k [B,1,h_qk,d_k]; v [B,1,h_v,d_v]; a, b [B,1,h_v];
    pool [P,h_v,d_k,d_v] fp32; slots int32 [B] on the device.  Returns o [B,1,h_v,d_v]."""
    lib = load()
    shape = _shape_of(q, v, None)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    _need_cuda("pool", pool, torch.float32)
    _need_cuda("slots", slots, torch.int32)
    if pool.dim() != 4 or tuple(pool.shape[1:]) != (shape.h_v, shape.d_k, shape.d_v):
        raise GdnError(GDN_ERR_INVALID_ARG, "pool must be [P, h_v, d_k, d_v]")
    if tuple(slots.shape) != (shape.batch,):
        raise GdnError(GDN_ERR_INVALID_ARG, "slots must be [B]")
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("o", o, dt)
    _check(lib.gdn_decode_step_slots(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                                     _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(pool),
                                     int(pool.shape[0]), _ptr(slots), float(scale), _ptr(o),
                                     _stream(stream)))
    return o


def gdn_scan_window(q, k, v, a, b, A_log, dt_bias, state_in=None, scale: float = 0.0, *,
                    window_len: int, o=None, window=None, stream=None):
    """Run B sequences of T tokens and return (o, window): window[w] is the state after
    step T - window_len + w, with zero slabs first when T < window_len.
    q, k [B,T,h_qk,d_k]; v [B,T,h_v,d_v]; a, b [B,T,h_v]; state_in [B,h_v,d_k,d_v] or None;
    window [window_len, B, h_v, d_k, d_v] fp32."""
    lib = load()
    shape = _shape_of(q, v, None)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("b", b)):
        _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    st_shape = (shape.batch, shape.h_v, shape.d_k, shape.d_v)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
        if tuple(state_in.shape) != st_shape:
            raise GdnError(GDN_ERR_INVALID_ARG, f"state_in must be {st_shape}")
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("o", o, dt)
    if window is None:
        window = torch.empty((int(window_len),) + st_shape, dtype=torch.float32, device=v.device)
    else:
        _need_cuda("window", window, torch.float32)
    _check(lib.gdn_scan_window(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(b),
                               _ptr(A_log), _ptr(dt_bias), _ptr(state_in), float(scale), _ptr(o),
                               _ptr(window), int(window_len), _stream(stream)))
    return o, window


def _variant_args(q, k, v, a, b, A_log, dt_bias, state_in, cu_seqlens, rule, decay_per_key,
                  beta_shared, o, state_out):
    """Validate a variant call; returns (shape, variant, o, state_out, the pointers a, b,
    A_log, dt_bias the rule reads)."""
    if rule not in RULES:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unknown rule {rule!r}")
    shape = _shape_of(q, v, cu_seqlens)
    dt = q.dtype
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, dt)
    if tuple(k.shape) != tuple(q.shape):
        raise GdnError(GDN_ERR_INVALID_ARG, "k must match q")
    lead = tuple(v.shape[:2])
    decay = rule in ("gated_delta", "gated")
    delta = rule in ("gated_delta", "delta")
    if decay:
        _need_cuda("a", a, dt)
        _need_cuda("A_log", A_log, torch.float32)
        _need_cuda("dt_bias", dt_bias, torch.float32)
        per = (shape.h_v, shape.d_k) if decay_per_key else (shape.h_v,)
        if tuple(a.shape) != lead + per or tuple(A_log.shape) != per or \
                tuple(dt_bias.shape) != per:
            raise GdnError(GDN_ERR_INVALID_ARG, f"a must be {lead + per}, A_log and dt_bias {per}")
    if delta:
        _need_cuda("b", b, dt)
        want = lead + ((1,) if beta_shared else (shape.h_v,))
        if tuple(b.shape) != want:
            raise GdnError(GDN_ERR_INVALID_ARG, f"b must be {want}")
    st_shape = (shape.num_seqs, shape.h_v, shape.d_k, shape.d_v)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
        if tuple(state_in.shape) != st_shape:
            raise GdnError(GDN_ERR_INVALID_ARG, f"state_in must be {st_shape}")
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    if o is None:
        o = torch.empty(v.shape, dtype=dt, device=v.device)
    else:
        _need_cuda("o", o, dt)
    if state_out is None:
        state_out = torch.empty(st_shape, dtype=torch.float32, device=v.device)
    else:
        _need_cuda("state_out", state_out, torch.float32)
    var = GdnVariant(RULES[rule], int(bool(decay_per_key)), int(bool(beta_shared)))
    gates = (_ptr(a if decay else None), _ptr(b if delta else None),
             _ptr(A_log if decay else None), _ptr(dt_bias if decay else None))
    return shape, var, o, state_out, gates


def gdn_scan_variant(q, k, v, a=None, b=None, A_log=None, dt_bias=None, state_in=None,
                     cu_seqlens=None, scale: float = 0.0, *, rule: str = "gated_delta",
                     decay_per_key: bool = False, beta_shared: bool = False, o=None,
                     state_out=None, stream=None):
    """gdn_prefill with another update rule ("gated_delta", "delta", "gated", "linear"),
    per-key-dim decay (a [B,T,h_v,d_k]; A_log, dt_bias [h_v,d_k]) or one beta for all
    heads (b [B,T,1]), on the token-sequential kernel.  a, A_log, dt_bias are unused (may
    be None) by rules without decay, b by rules without the delta term.  Returns
    (o, state_out); ``state_out`` may be ``state_in`` itself (an in-place update)."""
    lib = load()
    shape, var, o, state_out, gates = _variant_args(q, k, v, a, b, A_log, dt_bias, state_in,
                                                    cu_seqlens, rule, decay_per_key, beta_shared,
                                                    o, state_out)
    _check(lib.gdn_scan_variant(ctypes.byref(shape), ctypes.byref(var), _ptr(q), _ptr(k), _ptr(v),
                                *gates, _ptr(state_in), _ptr(cu_seqlens), float(scale), _ptr(o),
                                _ptr(state_out), _stream(stream)))
    return o, state_out


def gdn_prefill_variant(q, k, v, a=None, b=None, A_log=None, dt_bias=None, state_in=None,
                        cu_seqlens=None, scale: float = 0.0, *, rule: str = "gated_delta",
                        decay_per_key: bool = False, beta_shared: bool = False, o=None,
                        state_out=None, workspace=None, stream=None):
    """gdn_scan_variant on gdn_prefill's path: the chunked tensor-core prefill for 16-bit
    I/O at d_k = d_v = 128 (any rule, shared or per-head beta, per-key-dim decay), the
    token-sequential kernel for other shapes.  ``workspace`` defaults to
    gdn_prefill_variant_workspace_bytes; a per-key decay given less (down to
    gdn_prefill_workspace_bytes) runs the token-sequential kernel."""
    lib = load()
    shape, var, o, state_out, gates = _variant_args(q, k, v, a, b, A_log, dt_bias, state_in,
                                                    cu_seqlens, rule, decay_per_key, beta_shared,
                                                    o, state_out)
    need = int(lib.gdn_prefill_variant_workspace_bytes(ctypes.byref(shape), ctypes.byref(var)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=v.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.gdn_prefill_variant(ctypes.byref(shape), ctypes.byref(var), _ptr(q), _ptr(k), _ptr(v),
                                   *gates, _ptr(state_in), _ptr(cu_seqlens), float(scale), _ptr(o),
                                   _ptr(state_out), _ptr(workspace), ws_bytes, _stream(stream)))
    return o, state_out


# ---------------------------------------------------------------- neighbouring ops

def _conv_geometry(x, weight, channels_last: bool):
    if x.dim() != 3:
        raise GdnError(GDN_ERR_INVALID_ARG, "x must be [B, L, C] (or [B, C, L])")
    if x.dtype not in _DTYPE_CODE:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unsupported io dtype {x.dtype}")
    B = x.shape[0]
    L, C = (x.shape[1], x.shape[2]) if channels_last else (x.shape[2], x.shape[1])
    if weight.numel() == 0 or weight.numel() % C != 0 or weight.shape[0] != C:
        raise GdnError(GDN_ERR_INVALID_ARG, "weight must be [C, 1, K] or [C, K, 1]")
    return B, L, C, weight.numel() // C


def conv_state_shape(B: int, C: int, K: int, dilation: int = 1, channels_last: bool = True,
                     state_window: int = 0):
    carry = (K - 1) * dilation
    shape = (B, carry, C) if channels_last else (B, C, carry)
    return ((state_window,) + shape) if state_window else shape


def gdn_causal_conv(x, weight, bias=None, state_in=None, *, dilation: int = 1,
                    channels_last: bool = True, activation: str = "none",
                    state_window: int = 0, y=None, state_out=None, stream=None):
    """Causal depthwise convolution with a carried state; returns (y, state_out).

    x [B, L, C] (channels_last) or [B, C, L]; weight [C, 1, K]; bias [C] or None;
    state_in [B, carry, C] / [B, C, carry] with a leading [W] axis when state_window = W,
    or None (zeros); carry = (K - 1) * dilation.  ``state_out`` may be ``state_in``."""
    lib = load()
    B, L, C, K = _conv_geometry(x, weight, channels_last)
    dt = x.dtype
    _need_cuda("x", x, dt)
    _need_cuda("weight", weight, dt)
    if bias is not None:
        _need_cuda("bias", bias, dt)
        if tuple(bias.shape) != (C,):
            raise GdnError(GDN_ERR_INVALID_ARG, f"bias must be [{C}]")
    st_shape = conv_state_shape(B, C, K, dilation, channels_last, state_window)
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None:
            _need_cuda(name, t, dt)
            if tuple(t.shape) != st_shape:
                raise GdnError(GDN_ERR_INVALID_ARG, f"{name} must be {st_shape}")
    if y is None:
        y = torch.empty(x.shape, dtype=dt, device=x.device)
    else:
        _need_cuda("y", y, dt)
    if state_out is None:
        state_out = torch.empty(st_shape, dtype=dt, device=x.device)
    shape = GdnConvShape(_DTYPE_CODE[dt], B, L, C, K, int(dilation), int(bool(channels_last)),
                         ACTIVATIONS[activation], int(state_window))
    _check(lib.gdn_causal_conv(ctypes.byref(shape), _ptr(x), _ptr(weight), _ptr(bias),
                               _ptr(state_in), _ptr(y), _ptr(state_out), _stream(stream)))
    return y, state_out


def gdn_causal_conv_slots(x, weight, pool, slots, bias=None, *, dilation: int = 1,
                          activation: str = "none", y=None, stream=None):
    """The convolution against a pool of states: row b reads and updates
    ``pool[slots[b]]`` in place.  x [B, L, C]; pool [P, carry, C]; slots int32 [B].
    Returns y [B, L, C]."""
    lib = load()
    B, L, C, K = _conv_geometry(x, weight, True)
    dt = x.dtype
    for name, t in (("x", x), ("weight", weight), ("pool", pool)):
        _need_cuda(name, t, dt)
    _need_cuda("slots", slots, torch.int32)
    carry = (K - 1) * dilation
    if pool.dim() != 3 or tuple(pool.shape[1:]) != (carry, C):
        raise GdnError(GDN_ERR_INVALID_ARG, f"pool must be [P, {carry}, {C}]")
    if tuple(slots.shape) != (B,):
        raise GdnError(GDN_ERR_INVALID_ARG, "slots must be [B]")
    if bias is not None:
        _need_cuda("bias", bias, dt)
    if y is None:
        y = torch.empty(x.shape, dtype=dt, device=x.device)
    else:
        _need_cuda("y", y, dt)
    shape = GdnConvShape(_DTYPE_CODE[dt], B, L, C, K, int(dilation), 1, ACTIVATIONS[activation], 0)
    _check(lib.gdn_causal_conv_slots(ctypes.byref(shape), _ptr(x), _ptr(weight), _ptr(bias),
                                     _ptr(pool), int(pool.shape[0]), _ptr(slots), _ptr(y),
                                     _stream(stream)))
    return y


def gdn_gated_rmsnorm(x, scale, gate, eps: float = 1e-5, activation: str = "silu", *, y=None,
                      stream=None):
    """y = x / sqrt(mean(x^2) + eps) * scale * act(gate) over rows of len(scale) values."""
    lib = load()
    dt = x.dtype
    if dt not in _DTYPE_CODE:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unsupported io dtype {dt}")
    for name, t in (("x", x), ("scale", scale), ("gate", gate)):
        _need_cuda(name, t, dt)
    width = scale.numel()
    if scale.dim() != 1 or width == 0 or x.numel() % width != 0 or gate.shape != x.shape:
        raise GdnError(GDN_ERR_INVALID_ARG, "scale must be [C] dividing x's size; gate like x")
    if y is None:
        y = torch.empty(x.shape, dtype=dt, device=x.device)
    else:
        _need_cuda("y", y, dt)
    _check(lib.gdn_gated_rmsnorm(_DTYPE_CODE[dt], x.numel() // width, width, _ptr(x), _ptr(scale),
                                 _ptr(gate), float(eps), ACTIVATIONS[activation], _ptr(y),
                                 _stream(stream)))
    return y


def gdn_decode_layer(x, conv_weight, conv_bias, conv_state_in, conv_state_out, a, b, A_log,
                     dt_bias, state, norm_scale, gate, *, h_qk: int, h_v: int, d_k: int = 128,
                     scale: float = 0.0, conv_activation: str = "silu",
                     norm_activation: str = "silu", eps: float = 1e-5, y=None, stream=None):
    """One decode token of the layer: causal conv over x [B, 1, C] (channels read as
    [q | k | v], C = 2 h_qk d_k + h_v d_v), the gated delta-rule step on state
    [B, h_v, d_k, d_v] (in place), then the gated RMS norm of o with norm_scale [d_v] and
    gate [B, 1, h_v, d_v].  conv_weight [C, 1, K]; conv_bias [C] or None; conv states
    [B, K - 1, C] (conv_state_in None = zeros; conv_state_out None = not written; the two
    may not overlap).  Returns y [B, 1, h_v, d_v]."""
    lib = load()
    dt = x.dtype
    if dt not in _DTYPE_CODE:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unsupported io dtype {dt}")
    for name, t in (("x", x), ("conv_weight", conv_weight), ("a", a), ("b", b),
                    ("norm_scale", norm_scale), ("gate", gate)):
        _need_cuda(name, t, dt)
    for name, t in (("conv_bias", conv_bias), ("conv_state_in", conv_state_in),
                    ("conv_state_out", conv_state_out)):
        if t is not None:
            _need_cuda(name, t, dt)
    _need_cuda("state", state, torch.float32)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    if x.dim() != 3 or x.shape[1] != 1:
        raise GdnError(GDN_ERR_INVALID_ARG, "x must be [B, 1, C]")
    B, C = x.shape[0], x.shape[2]
    d_v = norm_scale.numel()
    if C != 2 * h_qk * d_k + h_v * d_v or conv_weight.numel() % C != 0:
        raise GdnError(GDN_ERR_INVALID_ARG, "x's channels must be 2 h_qk d_k + h_v d_v; weight [C, 1, K]")
    K = conv_weight.numel() // C
    if y is None:
        y = torch.empty((B, 1, h_v, d_v), dtype=dt, device=x.device)
    else:
        _need_cuda("y", y, dt)
    shape = make_shape(_DTYPE_CODE[dt], B, 1, B, h_qk, h_v, d_k, d_v)
    layer = GdnLayerParams(K, ACTIVATIONS[conv_activation], ACTIVATIONS[norm_activation], float(eps))
    _check(lib.gdn_decode_layer(ctypes.byref(shape), ctypes.byref(layer), _ptr(x), _ptr(conv_weight),
                                _ptr(conv_bias), _ptr(conv_state_in), _ptr(conv_state_out), _ptr(a),
                                _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(state), float(scale),
                                _ptr(norm_scale), _ptr(gate), _ptr(y), _stream(stream)))
    return y


def gdn_prefill_layer(x, conv_weight, conv_bias, conv_state_in, a, b, A_log, dt_bias, state_in,
                      cu_seqlens, norm_scale, gate, *, h_qk: int, h_v: int, scale: float = 0.0,
                      conv_activation: str = "silu", norm_activation: str = "silu", eps: float = 1e-5,
                      fuse: bool = False, y=None, state_out=None, conv_state_out=None, workspace=None,
                      stream=None):
    """The prefill of a layer: causal conv over x (channels [q | k | v], C = 2 h_qk 128 +
    h_v 128; [B, T, C], or [1, total, C] packed with cu_seqlens), the chunked prefill on its
    q, k, v, then the gated RMS norm of o.  conv_weight [C, 1, K] (K <= 4); conv_bias [C] or
    None; conv_state_in [N, K - 1, C] or None (zeros).  Returns (y [.., h_v, 128],
    state_out [N, h_v, 128, 128], conv_state_out [N, K - 1, C])."""
    lib = load()
    dt = x.dtype
    if dt not in _DTYPE_CODE:
        raise GdnError(GDN_ERR_INVALID_ARG, f"unsupported io dtype {dt}")
    for name, t in (("x", x), ("conv_weight", conv_weight), ("a", a), ("b", b),
                    ("norm_scale", norm_scale), ("gate", gate)):
        _need_cuda(name, t, dt)
    for name, t in (("conv_bias", conv_bias), ("conv_state_in", conv_state_in)):
        if t is not None:
            _need_cuda(name, t, dt)
    _need_cuda("A_log", A_log, torch.float32)
    _need_cuda("dt_bias", dt_bias, torch.float32)
    if x.dim() != 3:
        raise GdnError(GDN_ERR_INVALID_ARG, "x must be [B, T, C]")
    B, T, C = x.shape
    d = 128
    if C != 2 * h_qk * d + h_v * d or conv_weight.numel() % C != 0:
        raise GdnError(GDN_ERR_INVALID_ARG, "x's channels must be 2 h_qk 128 + h_v 128; weight [C, 1, K]")
    K = conv_weight.numel() // C
    if cu_seqlens is not None:
        _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
        if B != 1:
            raise GdnError(GDN_ERR_INVALID_ARG, "packed sequences need x [1, total, C]")
        n_seq = cu_seqlens.numel() - 1
        shape = make_shape(_DTYPE_CODE[dt], 1, T, n_seq, h_qk, h_v, d, d)
    else:
        n_seq = B
        shape = make_shape(_DTYPE_CODE[dt], B, T, B, h_qk, h_v, d, d)
    if state_in is not None:
        _need_cuda("state_in", state_in, torch.float32)
    if y is None:
        y = torch.empty((B, T, h_v, d), dtype=dt, device=x.device)
    if state_out is None:
        state_out = torch.empty((n_seq, h_v, d, d), dtype=torch.float32, device=x.device)
    if conv_state_out is None:
        conv_state_out = torch.empty((n_seq, max(K - 1, 0), C), dtype=dt, device=x.device)
    need = int(lib.gdn_prefill_layer_workspace_bytes(ctypes.byref(shape)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    layer = GdnLayerParams(K, ACTIVATIONS[conv_activation], ACTIVATIONS[norm_activation], float(eps))
    _check(lib.gdn_prefill_layer(ctypes.byref(shape), ctypes.byref(layer), _ptr(x), _ptr(conv_weight),
                                 _ptr(conv_bias), _ptr(conv_state_in), _ptr(conv_state_out), _ptr(a),
                                 _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(state_in), _ptr(cu_seqlens),
                                 float(scale), _ptr(norm_scale), _ptr(gate), _ptr(y), _ptr(state_out),
                                 int(bool(fuse)), _ptr(workspace), ws_bytes, _stream(stream)))
    return y, state_out, conv_state_out
