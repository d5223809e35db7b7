"""CPU oracle for the gated delta-rule scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``gdn_ref.c`` (plain sequential
float64 C, built with gcc into ``oracle/_build/``) through ctypes.  It does not
import, link or share anything with the CUDA library.

Pins: every function here is checked in ``tests/test_oracle.py`` against facts
fixed independently of it -- a worked example printed on the onnxruntime-ep-mlx
ssm.rs page (``tests/golden/``), closed forms, invariants and a brute-force
product of transition matrices.  None is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_ref.c")
_SRCS = (_SRC, os.path.join(_HERE, "neighbours_ref.c"))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_ref.so")

RULES = {"gated_delta": 0, "delta": 1, "gated": 2, "linear": 3}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            any(os.path.getmtime(_LIB_PATH) < os.path.getmtime(src) for src in _SRCS):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                        "-pthread", *_SRCS, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        D = ctypes.POINTER(ctypes.c_double)
        I64 = ctypes.POINTER(ctypes.c_int64)
        lib.gdn_ref_scan.restype = ctypes.c_int
        lib.gdn_ref_scan.argtypes = [
            ctypes.c_int64, I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, D, D, D, D, D, D, D, D, D, D, ctypes.c_double,
            ctypes.c_int32, I64, ctypes.c_int64, ctypes.c_int32, D, D]
        lib.gdn_ref_scan_ex.restype = ctypes.c_int
        lib.gdn_ref_scan_ex.argtypes = [
            ctypes.c_int64, I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_int32, D, D, D, D, D, D, D, D, D, D, ctypes.c_double,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, I64, ctypes.c_int64, ctypes.c_int32,
            D, D]
        for name in ("gdn_ref_softplus", "gdn_ref_sigmoid"):
            getattr(lib, name).restype = ctypes.c_double
            getattr(lib, name).argtypes = [ctypes.c_double]
        lib.gdn_ref_decay.restype = ctypes.c_double
        lib.gdn_ref_decay.argtypes = [ctypes.c_double] * 3
        I32 = ctypes.c_int32
        lib.gdn_ref_causal_conv.restype = ctypes.c_int
        lib.gdn_ref_causal_conv.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, I32,
                                            I32, I32, I32, I32, D, D, D, D, D, D]
        lib.gdn_ref_gated_rmsnorm.restype = ctypes.c_int
        lib.gdn_ref_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int64, D, D, D,
                                              ctypes.c_double, I32, D]
        _lib = lib
    return _lib


def _ptr(x: Optional[np.ndarray], ctype=ctypes.c_double):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))


def softplus(x: float) -> float:
    return _load().gdn_ref_softplus(float(x))


def sigmoid(x: float) -> float:
    return _load().gdn_ref_sigmoid(float(x))


def decay(a: float, A_log: float, dt_bias: float) -> float:
    """g = -exp(A_log) * softplus(a + dt_bias)."""
    return _load().gdn_ref_decay(float(a), float(A_log), float(dt_bias))


def scan(cu_seqlens: Sequence[int], h_qk: int, h_v: int, d_k: int, d_v: int,
         q, k, v, a=None, b=None, A_log=None, dt_bias=None, g=None, beta=None,
         state_in=None, scale: Optional[float] = None, rule: str = "gated_delta",
         units: Optional[Sequence[int]] = None, threads: int = 1,
         decay_per_key: bool = False, beta_shared: bool = False):
    """Run the recurrence over packed tokens.

    q, k: [T_total, h_qk, d_k]; v: [T_total, h_v, d_v]; a, b, g, beta: [T_total, h_v];
    A_log, dt_bias: [h_v]; state_in: [n_seq, h_v, d_k, d_v] or None.
    If ``a`` is None the gates are ``g`` (log-space, None = 0) and ``beta``
    (None = 1).  ``scale`` None means 1/sqrt(d_k).  ``units`` restricts the run
    to the listed (n * h_v + h) units; other rows of the outputs stay zero.
    ``decay_per_key``: a (or g) is [T_total, h_v, d_k] and A_log, dt_bias are
    [h_v, d_k] -- row i of the state decays by its own factor.  ``beta_shared``: b
    (or beta) is [T_total], one beta for all heads.
    Returns (o [T_total, h_v, d_v], state_out [n_seq, h_v, d_k, d_v]) in float64.
    """
    lib = _load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    n_seq = len(cu) - 1
    total = int(cu[-1]) if n_seq >= 0 and len(cu) else 0
    if scale is None or scale == 0.0:
        scale = 1.0 / np.sqrt(d_k)
    q, k, v = _f64(q), _f64(k), _f64(v)
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    g, beta, state_in = _f64(g), _f64(beta), _f64(state_in)
    assert q.size == total * h_qk * d_k and k.size == q.size
    assert v.size == total * h_v * d_v
    o = np.zeros(total * h_v * d_v, dtype=np.float64)
    s_out = np.zeros(max(n_seq, 0) * h_v * d_k * d_v, dtype=np.float64)
    ulist = None if units is None else np.ascontiguousarray(np.asarray(units, dtype=np.int64))
    rc = lib.gdn_ref_scan_ex(
        n_seq, _ptr(cu, ctypes.c_int64), h_qk, h_v, d_k, d_v, _ptr(q), _ptr(k), _ptr(v),
        _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias), _ptr(g), _ptr(beta), _ptr(state_in),
        float(scale), RULES[rule], int(bool(decay_per_key)), int(bool(beta_shared)),
        _ptr(ulist, ctypes.c_int64), 0 if ulist is None else len(ulist), int(threads), _ptr(o),
        _ptr(s_out))
    if rc != 0:
        raise ValueError(f"gdn_ref_scan_ex failed with code {rc}")
    return o.reshape(total, h_v, d_v), s_out.reshape(max(n_seq, 0), h_v, d_k, d_v)


def scan_inputs(inp, units=None, threads: int = 1, rule: Optional[str] = None):
    """Run the oracle on a drawn ``workloads.Inputs`` (the float64 copies), with the
    spec's gate layout (per-key decay, shared beta) and update rule (``rule`` overrides
    it)."""
    s = inp.spec
    f = inp.f64
    rule = rule or getattr(s, "rule", "gated_delta")
    return scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"],
                a=f["a"], b=f["b"], A_log=f["A_log"], dt_bias=f["dt_bias"],
                state_in=f["state_in"], scale=inp.scale, rule=rule, units=units,
                threads=threads, decay_per_key=s.decay_per_key, beta_shared=s.beta_shared)


def slot_scan(cu_seqlens: Sequence[int], h_qk: int, h_v: int, d_k: int, d_v: int,
              q, k, v, a, b, A_log, dt_bias, pool, slots, scale: Optional[float] = None,
              threads: int = 1):
    """The rule against a pool of states (nuvec-core src/fast/imp.rs, `gated_delta_slots`
    and the fallback graph of FastOp::GatedDeltaSlots): take the states at the slots, run
    the recurrence, put the new states back at the slots.

    pool: [P, h_v, d_k, d_v]; slots: [n_seq] integers.  Sequence n starts from
    pool[slots[n]] and its final state is written there; entries not named by a slot are
    unchanged.  A slot outside [0, P) -- which the pages leave open -- skips its
    sequence: its outputs stay zero and the pool is unchanged.  With repeated slots the
    later sequence's state lands last.  Returns (o, new pool) in float64.
    """
    pool = np.array(_f64(pool), dtype=np.float64, copy=True).reshape(-1, h_v, d_k, d_v)
    P = pool.shape[0]
    slots = [int(x) for x in np.asarray(slots).reshape(-1)]
    n_seq = len(cu_seqlens) - 1
    assert len(slots) == n_seq
    taken = np.zeros((n_seq, h_v, d_k, d_v), dtype=np.float64)
    kept = [n for n in range(n_seq) if 0 <= slots[n] < P]
    for n in kept:
        taken[n] = pool[slots[n]]
    units = [n * h_v + h for n in kept for h in range(h_v)]
    o, s_out = scan(cu_seqlens, h_qk, h_v, d_k, d_v, q, k, v, a=a, b=b, A_log=A_log,
                    dt_bias=dt_bias, state_in=taken, scale=scale, units=units, threads=threads)
    for n in kept:
        pool[slots[n]] = s_out[n]
    return o, pool


def slot_scan_inputs(inp, threads: int = 1):
    """slot_scan on a drawn ``workloads.Inputs`` that carries a pool and slots."""
    s = inp.spec
    f = inp.f64
    return slot_scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"],
                     f["a"], f["b"], f["A_log"], f["dt_bias"], f["pool"], inp.slots.numpy(),
                     scale=inp.scale, threads=threads)


def window_scan(batch: int, seqlen: int, h_qk: int, h_v: int, d_k: int, d_v: int, q, k, v,
                a, b, A_log, dt_bias, state_in, window_len: int, scale: Optional[float] = None,
                threads: int = 1):
    """The recurrence over B sequences of T tokens, keeping the states after the last
    `window_len` steps (onnxruntime-ep-mlx ssm.rs, LinearAttention `state_window`: the
    last min(T, W) step states in time order, after W - min(T, W) zero slabs).  Each step
    is one call of `scan` on a single token, chained through its state.

    Returns (o [B*T, h_v, d_v], window [W, B, h_v, d_k, d_v]) in float64.
    """
    B, T, W = int(batch), int(seqlen), int(window_len)
    q = _f64(q).reshape(B, T, h_qk, d_k)
    k = _f64(k).reshape(B, T, h_qk, d_k)
    v = _f64(v).reshape(B, T, h_v, d_v)
    a = _f64(a).reshape(B, T, h_v)
    b = _f64(b).reshape(B, T, h_v)
    state = (np.zeros((B, h_v, d_k, d_v)) if state_in is None
             else _f64(state_in).reshape(B, h_v, d_k, d_v).copy())
    o = np.zeros((B, T, h_v, d_v))
    window = np.zeros((W, B, h_v, d_k, d_v))
    cu1 = np.arange(B + 1)
    for t in range(T):
        o_t, state = scan(cu1, h_qk, h_v, d_k, d_v, q[:, t], k[:, t], v[:, t], a=a[:, t],
                          b=b[:, t], A_log=A_log, dt_bias=dt_bias, state_in=state, scale=scale,
                          threads=threads)
        o[:, t] = o_t
        w = W - (T - t)
        if w >= 0:
            window[w] = state
    return o.reshape(B * T, h_v, d_v), window


def window_scan_inputs(inp, threads: int = 1):
    """window_scan on a drawn ``workloads.Inputs`` whose spec sets a window."""
    s = inp.spec
    f = inp.f64
    return window_scan(s.batch, s.seqlen, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"],
                       f["a"], f["b"], f["A_log"], f["dt_bias"], f["state_in"], s.window,
                       scale=inp.scale, threads=threads)


# ---------------------------------------------------------------- neighbouring ops

ACTIVATIONS = {"silu": 1, "swish": 1, "sigmoid": 2}


def causal_conv(x, w, bias=None, state_in=None, *, dilation: int = 1,
                channels_last: bool = True, silu: bool = False, state_window: int = 0):
    """CausalConvWithState (onnxruntime-ep-mlx src/ops/ssm.rs, `causal_conv_op`).

    x: [B, L, C] (channels_last) or [B, C, L]; w: [C, 1, K] (or [C, K, 1], the same
    memory); bias: [C] or None; state_in: [B, carry, C] / [B, C, carry], with a leading
    [W] axis when state_window = W > 0, or None (zeros); carry = (K - 1) * dilation.
    Returns (y like x, state_out like state_in) in float64.
    """
    x = np.asarray(x, dtype=np.float64)
    B = x.shape[0]
    C = x.shape[2] if channels_last else x.shape[1]
    L = x.shape[1] if channels_last else x.shape[2]
    w = _f64(w)
    K = w.size // C
    assert K * C == w.size
    carry = (K - 1) * dilation
    st_shape = (B, carry, C) if channels_last else (B, C, carry)
    if state_window:
        st_shape = (state_window,) + st_shape
    if state_in is not None:
        assert np.size(state_in) == int(np.prod(st_shape))
    y = np.zeros(B * L * C, dtype=np.float64)
    s_out = np.zeros(int(np.prod(st_shape)), dtype=np.float64)
    rc = _load().gdn_ref_causal_conv(B, L, C, K, dilation, int(bool(channels_last)),
                                     int(bool(silu)), int(state_window), _ptr(_f64(x)), _ptr(w),
                                     _ptr(_f64(bias)), _ptr(_f64(state_in)), _ptr(y), _ptr(s_out))
    if rc != 0:
        raise ValueError(f"gdn_ref_causal_conv failed with code {rc}")
    return y.reshape(x.shape), s_out.reshape(st_shape)


def conv_slots(x, w, pool, slots, bias=None, *, dilation: int = 1, silu: bool = False):
    """The convolution against a pool of states (nuvec-core src/fast/imp.rs,
    `causal_conv1d_slots` and the fallback graph of FastOp::ConvSlots): take the states
    at the slots, prepend them to x [B, L, C], convolve, and put each row's last carry
    inputs back at its slot.  pool: [P, carry, C].  A slot outside [0, P) skips its row
    (outputs zero, pool unchanged).  Returns (y, new pool) in float64."""
    x = np.asarray(x, dtype=np.float64)
    B, L, C = x.shape
    pool = np.array(pool, dtype=np.float64, copy=True)
    P = pool.shape[0]
    y = np.zeros_like(x)
    for b, s in enumerate(int(v) for v in np.asarray(slots).reshape(-1)):
        if not 0 <= s < P:
            continue
        yb, sb = causal_conv(x[b:b + 1], w, bias, pool[s:s + 1], dilation=dilation, silu=silu)
        y[b] = yb[0]
        pool[s] = sb[0]
    return y, pool


def gated_rmsnorm(x, scale, gate, eps: float = 1e-5, activation: str = "silu"):
    """GatedRMSNorm (onnxruntime-ep-mlx src/ops/ssm.rs, `gated_rms_norm_op`): rows of
    C = len(scale) consecutive values of x.  Returns y (shape of x) in float64."""
    x = np.asarray(x, dtype=np.float64)
    scale = _f64(scale)
    width = scale.size
    assert x.size % width == 0 and np.size(gate) == x.size
    y = np.zeros(x.size, dtype=np.float64)
    rc = _load().gdn_ref_gated_rmsnorm(x.size // width, width, _ptr(_f64(x)), _ptr(scale),
                                       _ptr(_f64(gate)), float(eps), ACTIVATIONS[activation],
                                       _ptr(y))
    if rc != 0:
        raise ValueError(f"gdn_ref_gated_rmsnorm failed with code {rc}")
    return y.reshape(x.shape)
