"""Seeded synthetic inputs for the gated delta-rule scan.

This module is shared by the tests, the benchmark and the CPU oracle's callers.
It holds none of the method's arithmetic: no gates, no decay, no recurrence.
It only draws random numbers, L2-normalises q and k per (token, head) as the
input recipe asks, and rounds the draws once to the I/O dtype.  The oracle is
then handed the widened float64 copies of exactly those rounded values, and
the GPU path the rounded tensors themselves, so both see the same bits.

Recipe (one numpy ``default_rng(seed)``, float64 draws in this order):
  (varlen only: the sequence lengths), q, k, v, a, b, A_log, dt_bias, state_in.
  q, k ~ N(0, 1) then divided by their L2 norm over d_k; v, a, b ~ N(0, 1);
  A_log ~ U(-1, 1) and dt_bias ~ N(0, 0.1) per value head (fp32);
  state_in ~ N(0, state_std) fp32 when the workload asks for one (std, not
  variance), else no draw and a zero state.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and distribution of one synthetic workload."""
    name: str
    io: str                      # "f32" | "bf16" | "f16": q,k,v,a,b,o dtype
    h_qk: int
    h_v: int
    d_k: int
    d_v: int
    seed: int
    batch: int = 1               # B for batched (non-varlen) input
    seqlen: int = 0              # T per sequence for batched input
    lengths: Optional[Sequence[int]] = None   # explicit varlen lengths
    varlen_range: Optional[tuple] = None      # (lo, hi) inclusive, drawn first
    n_varlen: int = 0
    state_std: float = 0.0       # 0 -> zero initial state (state_in = None)
    decode: bool = False         # one token per sequence, state updated in place
    qk_scale: float = 1.0        # multiplies q,k after normalisation (tests only)
    pool_size: int = 0           # > 0: states live in a pool of this many entries
    pool_std: float = 0.0        # std of the pool entries
    window: int = 0              # > 0: emit the states after the last `window` steps
    decay_per_key: bool = False  # a [B,T,h_v,d_k], A_log and dt_bias [h_v,d_k]
    beta_shared: bool = False    # b [B,T,1]: one beta for every head
    rule: str = "gated_delta"    # the update rule (gated_delta, delta, gated, linear)


# The five workloads the method is measured on.
WORKLOADS = {
    "tiny_f32_prefill": Spec(
        "tiny_f32_prefill", io="f32", batch=1, seqlen=64, h_qk=2, h_v=2,
        d_k=32, d_v=32, seed=1000),
    "bf16_prefill_t4096": Spec(
        "bf16_prefill_t4096", io="bf16", batch=1, seqlen=4096, h_qk=16, h_v=16,
        d_k=128, d_v=128, seed=1001),
    "bf16_decode_b256": Spec(
        "bf16_decode_b256", io="bf16", batch=256, seqlen=1, h_qk=32, h_v=32,
        d_k=128, d_v=128, seed=1002, state_std=0.05, decode=True),
    "varlen_bf16_prefill": Spec(
        "varlen_bf16_prefill", io="bf16", h_qk=16, h_v=16, d_k=128, d_v=128,
        seed=1003, varlen_range=(512, 8192), n_varlen=8, state_std=0.05),
    "gqa_f16_prefill": Spec(
        "gqa_f16_prefill", io="f16", batch=2, seqlen=8192, h_qk=16, h_v=32,
        d_k=128, d_v=128, seed=1004),
    # Decode against a pool of 512 states, 256 sequences at distinct slots (the slot-pool
    # decode row that follows the five above).
    "bf16_slot_decode_b256": Spec(
        "bf16_slot_decode_b256", io="bf16", batch=256, seqlen=1, h_qk=32, h_v=32,
        d_k=128, d_v=128, seed=1005, decode=True, pool_size=512, pool_std=0.05),
    # Speculative verify: 4 draft tokens for each of 256 sequences, emitting the state
    # after every step (the per-step-state row).
    "bf16_window_b256_t4": Spec(
        "bf16_window_b256_t4", io="bf16", batch=256, seqlen=4, h_qk=32, h_v=32,
        d_k=128, d_v=128, seed=1006, state_std=0.05, window=4),
    # Decode with one decay per key dimension (the gate-variant row).
    "bf16_perkey_decode_b256": Spec(
        "bf16_perkey_decode_b256", io="bf16", batch=256, seqlen=1, h_qk=32, h_v=32,
        d_k=128, d_v=128, seed=1007, state_std=0.05, decode=True, decay_per_key=True),
    # The gate-variant row at prefill length, on the 4,096-token shape: the delta rule and
    # one shared beta run on the chunked tensor-core path, per-key decay on the
    # token-sequential kernel.
    "bf16_delta_prefill_t4096": Spec(
        "bf16_delta_prefill_t4096", io="bf16", batch=1, seqlen=4096, h_qk=16, h_v=16,
        d_k=128, d_v=128, seed=1008, rule="delta"),
    "bf16_shared_beta_prefill_t4096": Spec(
        "bf16_shared_beta_prefill_t4096", io="bf16", batch=1, seqlen=4096, h_qk=16, h_v=16,
        d_k=128, d_v=128, seed=1009, beta_shared=True),
    "bf16_perkey_prefill_t4096": Spec(
        "bf16_perkey_prefill_t4096", io="bf16", batch=1, seqlen=4096, h_qk=16, h_v=16,
        d_k=128, d_v=128, seed=1015, decay_per_key=True),
}


@dataclasses.dataclass
class Inputs:
    """One drawn workload.  Torch tensors live on the CPU in their final dtype;
    ``f64`` holds float64 copies (widened from those exact values) for the oracle."""
    spec: Spec
    cu_seqlens: np.ndarray        # int64 [n_seq+1] token offsets into the packed axis
    q: torch.Tensor               # [B, T, h_qk, d_k] (varlen: B=1, T=total)
    k: torch.Tensor
    v: torch.Tensor               # [B, T, h_v, d_v]
    a: torch.Tensor               # [B, T, h_v] ([B, T, h_v, d_k] with decay_per_key)
    b: torch.Tensor               # [B, T, h_v] ([B, T, 1] with beta_shared)
    A_log: torch.Tensor           # [h_v] fp32 ([h_v, d_k] with decay_per_key)
    dt_bias: torch.Tensor         # [h_v] fp32 ([h_v, d_k] with decay_per_key)
    state_in: Optional[torch.Tensor]   # [n_seq, h_v, d_k, d_v] fp32 or None
    scale: float
    f64: dict
    pool: Optional[torch.Tensor] = None    # [pool_size, h_v, d_k, d_v] fp32
    slots: Optional[torch.Tensor] = None   # int32 [n_seq], distinct entries of the pool

    @property
    def n_seq(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def varlen(self) -> bool:
        return self.spec.lengths is not None or self.spec.varlen_range is not None

    def lengths(self) -> np.ndarray:
        return np.diff(self.cu_seqlens)


def _round(x: np.ndarray, io: str) -> torch.Tensor:
    """Round float64 draws once, to nearest even, into the given dtype."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(_TORCH_DTYPE[io])


def _widen(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy().reshape(-1)


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.where(n == 0.0, 1.0, n)


def draw(spec: Spec) -> Inputs:
    """Draw the inputs of ``spec`` with its seed, in the recipe's order."""
    rng = np.random.default_rng(spec.seed)
    if spec.varlen_range is not None:
        lo, hi = spec.varlen_range
        lengths = rng.integers(lo, hi + 1, spec.n_varlen)
    elif spec.lengths is not None:
        lengths = np.asarray(spec.lengths, dtype=np.int64)
    else:
        lengths = None
    if lengths is not None:
        B, T = 1, int(np.sum(lengths))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    else:
        B, T = spec.batch, spec.seqlen
        cu = np.arange(B + 1, dtype=np.int64) * T
    n_seq = len(cu) - 1

    q = _l2_normalise(rng.standard_normal((B, T, spec.h_qk, spec.d_k))) * spec.qk_scale
    k = _l2_normalise(rng.standard_normal((B, T, spec.h_qk, spec.d_k))) * spec.qk_scale
    v = rng.standard_normal((B, T, spec.h_v, spec.d_v))
    per = (spec.h_v, spec.d_k) if spec.decay_per_key else (spec.h_v,)
    a = rng.standard_normal((B, T) + per)
    b = rng.standard_normal((B, T, 1 if spec.beta_shared else spec.h_v))
    A_log = rng.uniform(-1.0, 1.0, per)
    dt_bias = rng.normal(0.0, 0.1, per)
    state = None
    if spec.state_std > 0.0:
        state = rng.normal(0.0, spec.state_std, (n_seq, spec.h_v, spec.d_k, spec.d_v))
    pool = slots = None
    if spec.pool_size > 0:
        pool = rng.normal(0.0, spec.pool_std, (spec.pool_size, spec.h_v, spec.d_k, spec.d_v))
        slots = rng.permutation(spec.pool_size)[:n_seq].astype(np.int32)

    tq, tk, tv = _round(q, spec.io), _round(k, spec.io), _round(v, spec.io)
    ta, tb = _round(a, spec.io), _round(b, spec.io)
    tA, tdt = _round(A_log, "f32"), _round(dt_bias, "f32")
    ts = None if state is None else _round(state, "f32")
    f64 = {
        "q": _widen(tq), "k": _widen(tk), "v": _widen(tv),
        "a": _widen(ta), "b": _widen(tb),
        "A_log": _widen(tA), "dt_bias": _widen(tdt),
        "state_in": None if ts is None else _widen(ts),
    }
    tp = tsl = None
    if pool is not None:
        tp = _round(pool, "f32")
        tsl = torch.from_numpy(slots)
        f64["pool"] = _widen(tp)
    return Inputs(spec=spec, cu_seqlens=cu, q=tq, k=tk, v=tv, a=ta, b=tb,
                  A_log=tA, dt_bias=tdt, state_in=ts,
                  scale=1.0 / math.sqrt(spec.d_k), f64=f64, pool=tp, slots=tsl)


def workload(name: str) -> Inputs:
    return draw(WORKLOADS[name])


def small_spec(name="small", io="bf16", batch=1, seqlen=0, lengths=None, h_qk=2,
               h_v=2, d_k=128, d_v=128, seed=7, state_std=0.0, decode=False,
               qk_scale=1.0, pool_size=0, pool_std=0.0, window=0, decay_per_key=False,
               beta_shared=False) -> Spec:
    """A test-sized workload with the same distributions as the measured ones."""
    return Spec(name=name, io=io, batch=batch, seqlen=seqlen,
                lengths=None if lengths is None else tuple(int(x) for x in lengths),
                h_qk=h_qk, h_v=h_v, d_k=d_k, d_v=d_v, seed=seed,
                state_std=state_std, decode=decode, qk_scale=qk_scale,
                pool_size=pool_size, pool_std=pool_std, window=window,
                decay_per_key=decay_per_key, beta_shared=beta_shared)


# ---------------------------------------------------------------- neighbouring ops
#
# The causal convolution that feeds q, k, v and the gated RMS norm of the scan's output.
# Recipe (one default_rng(seed), float64 draws in this order): x ~ N(0, 1); the weight
# ~ U(-1/sqrt(K), 1/sqrt(K)) (a depthwise conv's fan-in is K); the bias (when asked)
# likewise; the past state ~ N(0, state_std) (state_std 0: none) -- a window of them when
# state_window > 0, or a pool of pool_size entries followed by the slots, the first B
# entries of a permutation of the pool.  The norm draws x ~ N(0, 1), the gate ~ N(0, 1)
# and the scale ~ N(1, 0.1).  Every draw is rounded once to the I/O dtype.

@dataclasses.dataclass(frozen=True)
class ConvSpec:
    name: str
    io: str
    batch: int
    seqlen: int
    channels: int
    seed: int
    kernel: int = 4
    dilation: int = 1
    channels_last: bool = True
    silu: bool = True
    bias: bool = False
    state_std: float = 0.0
    state_window: int = 0
    pool_size: int = 0
    decode: bool = False         # one token per row, the state updated in place


@dataclasses.dataclass
class ConvInputs:
    spec: ConvSpec
    x: torch.Tensor               # [B, L, C] (channels first: [B, C, L])
    w: torch.Tensor               # [C, 1, K]
    bias: Optional[torch.Tensor]  # [C]
    state_in: Optional[torch.Tensor]   # [(W,) B, carry, C] / [(W,) B, C, carry]
    pool: Optional[torch.Tensor]       # [pool_size, carry, C]
    slots: Optional[torch.Tensor]      # int32 [B]
    f64: dict


@dataclasses.dataclass(frozen=True)
class NormSpec:
    name: str
    io: str
    shape: tuple                 # x's shape; the last dimension is the row width
    seed: int
    eps: float = 1e-6
    activation: str = "silu"


@dataclasses.dataclass
class NormInputs:
    spec: NormSpec
    x: torch.Tensor
    scale: torch.Tensor
    gate: torch.Tensor
    f64: dict


def draw_conv(spec: ConvSpec) -> ConvInputs:
    rng = np.random.default_rng(spec.seed)
    B, L, C, K = spec.batch, spec.seqlen, spec.channels, spec.kernel
    carry = (K - 1) * spec.dilation
    x = rng.standard_normal((B, L, C) if spec.channels_last else (B, C, L))
    lim = 1.0 / math.sqrt(K)
    w = rng.uniform(-lim, lim, (C, 1, K))
    bias = rng.uniform(-lim, lim, C) if spec.bias else None
    st_one = (B, carry, C) if spec.channels_last else (B, C, carry)
    state = pool = slots = None
    if spec.pool_size > 0:
        pool = rng.normal(0.0, spec.state_std, (spec.pool_size, carry, C))
        slots = rng.permutation(spec.pool_size)[:B].astype(np.int32)
    elif spec.state_std > 0.0:
        shape = ((spec.state_window,) + st_one) if spec.state_window else st_one
        state = rng.normal(0.0, spec.state_std, shape)
    t = {n: (None if a is None else _round(a, spec.io))
         for n, a in (("x", x), ("w", w), ("bias", bias), ("state_in", state), ("pool", pool))}
    f64 = {n: (None if v is None else _widen(v).reshape(v.shape)) for n, v in t.items()}
    return ConvInputs(spec=spec, x=t["x"], w=t["w"], bias=t["bias"], state_in=t["state_in"],
                      pool=t["pool"], slots=None if slots is None else torch.from_numpy(slots),
                      f64=f64)


def draw_norm(spec: NormSpec) -> NormInputs:
    rng = np.random.default_rng(spec.seed)
    x = rng.standard_normal(spec.shape)
    gate = rng.standard_normal(spec.shape)
    scale = rng.normal(1.0, 0.1, spec.shape[-1])
    t = {"x": _round(x, spec.io), "gate": _round(gate, spec.io), "scale": _round(scale, spec.io)}
    f64 = {n: _widen(v).reshape(v.shape) for n, v in t.items()}
    return NormInputs(spec=spec, x=t["x"], scale=t["scale"], gate=t["gate"], f64=f64)


# The measured neighbour workloads.  Channels: q, k, v side by side, at the GQA prefill's
# head counts (2 x 16 x 128 + 32 x 128 = 8192) and the decode step's (3 x 32 x 128 = 12288).
CONV_WORKLOADS = {
    "bf16_conv_prefill_gqa": ConvSpec(
        "bf16_conv_prefill_gqa", io="bf16", batch=2, seqlen=8192, channels=8192, seed=1010,
        state_std=1.0),
    "bf16_conv_decode_b256": ConvSpec(
        "bf16_conv_decode_b256", io="bf16", batch=256, seqlen=1, channels=12288, seed=1011,
        state_std=1.0, decode=True),
}
NORM_WORKLOADS = {
    # The scan output of the GQA prefill, [2, 8192, 32, 128], normalised per head.
    "bf16_norm_gqa": NormSpec("bf16_norm_gqa", io="bf16", shape=(2, 8192, 32, 128), seed=1012),
}


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """One decode token of the whole layer: conv over [q | k | v] channels, the step,
    the gated RMS norm."""
    name: str
    io: str
    batch: int
    h_qk: int
    h_v: int
    seed: int
    d_v: int = 128
    kernel: int = 4
    bias: bool = False
    conv_state_std: float = 1.0
    state_std: float = 0.05
    eps: float = 1e-6


@dataclasses.dataclass
class LayerInputs:
    spec: LayerSpec
    x: torch.Tensor               # [B, 1, C], C = 2 h_qk 128 + h_v d_v
    w: torch.Tensor               # [C, 1, K]
    bias: Optional[torch.Tensor]  # [C]
    conv_state: torch.Tensor      # [B, K - 1, C]
    a: torch.Tensor               # [B, 1, h_v]
    b: torch.Tensor
    A_log: torch.Tensor           # [h_v] fp32
    dt_bias: torch.Tensor
    state: torch.Tensor           # [B, h_v, 128, d_v] fp32
    norm_scale: torch.Tensor      # [d_v]
    gate: torch.Tensor            # [B, 1, h_v, d_v]
    f64: dict


def draw_layer(spec: LayerSpec) -> LayerInputs:
    rng = np.random.default_rng(spec.seed)
    B, K = spec.batch, spec.kernel
    C = 2 * spec.h_qk * 128 + spec.h_v * spec.d_v
    x = rng.standard_normal((B, 1, C))
    lim = 1.0 / math.sqrt(K)
    w = rng.uniform(-lim, lim, (C, 1, K))
    bias = rng.uniform(-lim, lim, C) if spec.bias else None
    conv_state = rng.normal(0.0, spec.conv_state_std, (B, K - 1, C))
    a = rng.standard_normal((B, 1, spec.h_v))
    b = rng.standard_normal((B, 1, spec.h_v))
    A_log = rng.uniform(-1.0, 1.0, spec.h_v)
    dt_bias = rng.normal(0.0, 0.1, spec.h_v)
    state = rng.normal(0.0, spec.state_std, (B, spec.h_v, 128, spec.d_v))
    norm_scale = rng.normal(1.0, 0.1, spec.d_v)
    gate = rng.standard_normal((B, 1, spec.h_v, spec.d_v))
    t = {n: (None if v is None else _round(v, spec.io))
         for n, v in (("x", x), ("w", w), ("bias", bias), ("conv_state", conv_state), ("a", a),
                      ("b", b), ("norm_scale", norm_scale), ("gate", gate))}
    t["A_log"] = _round(A_log, "f32")
    t["dt_bias"] = _round(dt_bias, "f32")
    t["state"] = _round(state, "f32")
    f64 = {n: (None if v is None else _widen(v).reshape(v.shape)) for n, v in t.items()}
    return LayerInputs(spec=spec, f64=f64, **t)


LAYER_WORKLOADS = {
    # The decode step's shape (B = 256, 32 heads, d = 128) with a 4-tap conv in front.
    "bf16_layer_decode_b256": LayerSpec("bf16_layer_decode_b256", io="bf16", batch=256, h_qk=32,
                                        h_v=32, seed=1013),
}


@dataclasses.dataclass(frozen=True)
class PrefillNormSpec:
    """A prefill workload whose output goes through the gated RMS norm (gdn_prefill_norm)."""
    name: str
    prefill: str                 # a WORKLOADS name
    seed: int
    eps: float = 1e-6
    activation: str = "silu"


@dataclasses.dataclass
class PrefillNormInputs:
    spec: PrefillNormSpec
    prefill: Inputs
    norm_scale: torch.Tensor     # [d_v]
    gate: torch.Tensor           # o's shape


def draw_prefill_norm(spec: PrefillNormSpec) -> PrefillNormInputs:
    inp = draw(WORKLOADS[spec.prefill])
    rng = np.random.default_rng(spec.seed)
    gate = rng.standard_normal(tuple(inp.v.shape))
    scale = rng.normal(1.0, 0.1, inp.spec.d_v)
    return PrefillNormInputs(spec=spec, prefill=inp, norm_scale=_round(scale, inp.spec.io),
                             gate=_round(gate, inp.spec.io))


PREFILL_NORM_WORKLOADS = {
    # The packed varlen prefill (8 sequences, 31,979 tokens, 16 heads, d = 128) with the
    # gated RMS norm of each head's output row.
    "varlen_bf16_prefill_norm": PrefillNormSpec("varlen_bf16_prefill_norm", "varlen_bf16_prefill",
                                                seed=1014),
}


@dataclasses.dataclass(frozen=True)
class PrefillLayerSpec:
    """The prefill of a whole layer (gdn_prefill_layer): the causal conv over the mixed
    input x [.., C] (C = 2 h_qk 128 + h_v 128, channels [q | k | v]), the chunked prefill
    on its q, k, v, then the gated RMS norm of o.

    Recipe (one default_rng(seed), float64 draws in this order, each rounded once to the
    I/O dtype, A_log / dt_bias / state to fp32): the lengths U[lo, hi] when varlen_range is
    set; x ~ N(0, x_std^2); the weight ~ U(-1/sqrt(K), 1/sqrt(K)); the bias likewise when
    asked; the conv state ~ N(0, 1); a, b ~ N(0, 1); A_log ~ U(-1, 1); dt_bias ~
    N(0, 0.1); the initial state ~ N(0, state_std^2) (0: none); the norm scale ~
    N(1, 0.1); the gate ~ N(0, 1).  The layer does not normalise q and k, so x_std = 0.3
    keeps the convolved keys' squared norm near 1 (about 128 x 0.3^2 / 12), where the
    delta rule's update I - beta k k^T stays contracting over thousands of tokens."""
    name: str
    io: str
    h_qk: int
    h_v: int
    seed: int
    batch: int = 1
    seqlen: int = 0
    lengths: Optional[tuple] = None
    varlen_range: Optional[tuple] = None
    n_varlen: int = 0
    kernel: int = 4
    bias: bool = True
    silu: bool = True
    x_std: float = 0.3
    state_std: float = 0.05
    eps: float = 1e-6
    activation: str = "silu"


@dataclasses.dataclass
class PrefillLayerInputs:
    spec: PrefillLayerSpec
    cu_seqlens: np.ndarray        # int64 [N + 1]
    x: torch.Tensor               # [B, T, C] (packed: [1, total, C])
    w: torch.Tensor               # [C, 1, K]
    bias: Optional[torch.Tensor]  # [C]
    conv_state: torch.Tensor      # [N, K - 1, C]
    a: torch.Tensor               # [B, T, h_v]
    b: torch.Tensor
    A_log: torch.Tensor           # [h_v] fp32
    dt_bias: torch.Tensor
    state_in: Optional[torch.Tensor]   # [N, h_v, 128, 128] fp32
    norm_scale: torch.Tensor      # [128]
    gate: torch.Tensor            # [B, T, h_v, 128]
    scale: float
    f64: dict

    @property
    def n_seq(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def varlen(self) -> bool:
        return self.spec.lengths is not None or self.spec.varlen_range is not None


def draw_prefill_layer(spec: PrefillLayerSpec) -> PrefillLayerInputs:
    rng = np.random.default_rng(spec.seed)
    if spec.varlen_range is not None:
        lo, hi = spec.varlen_range
        lengths = rng.integers(lo, hi + 1, spec.n_varlen)
    elif spec.lengths is not None:
        lengths = np.asarray(spec.lengths, dtype=np.int64)
    else:
        lengths = None
    if lengths is not None:
        B, T = 1, int(np.sum(lengths))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    else:
        B, T = spec.batch, spec.seqlen
        cu = np.arange(B + 1, dtype=np.int64) * T
    N, K = len(cu) - 1, spec.kernel
    C = 2 * spec.h_qk * 128 + spec.h_v * 128
    x = rng.normal(0.0, spec.x_std, (B, T, C))
    lim = 1.0 / math.sqrt(K)
    w = rng.uniform(-lim, lim, (C, 1, K))
    bias = rng.uniform(-lim, lim, C) if spec.bias else None
    conv_state = rng.normal(0.0, 1.0, (N, K - 1, C))
    a = rng.standard_normal((B, T, spec.h_v))
    b = rng.standard_normal((B, T, spec.h_v))
    A_log = rng.uniform(-1.0, 1.0, spec.h_v)
    dt_bias = rng.normal(0.0, 0.1, spec.h_v)
    state = rng.normal(0.0, spec.state_std, (N, spec.h_v, 128, 128)) if spec.state_std > 0 else None
    norm_scale = rng.normal(1.0, 0.1, 128)
    gate = rng.standard_normal((B, T, spec.h_v, 128))
    t = {n: (None if v is None else _round(v, spec.io))
         for n, v in (("x", x), ("w", w), ("bias", bias), ("conv_state", conv_state), ("a", a),
                      ("b", b), ("norm_scale", norm_scale), ("gate", gate))}
    t["A_log"] = _round(A_log, "f32")
    t["dt_bias"] = _round(dt_bias, "f32")
    t["state_in"] = None if state is None else _round(state, "f32")
    f64 = {n: (None if v is None else _widen(v).reshape(v.shape)) for n, v in t.items()}
    return PrefillLayerInputs(spec=spec, cu_seqlens=cu, scale=1.0 / math.sqrt(128), f64=f64, **t)


PREFILL_LAYER_WORKLOADS = {
    # The packed varlen prefill's shape (8 sequences drawn from U[512, 8192], 16 heads,
    # d = 128) with a 4-tap conv (bias, silu) in front and the gated norm after.
    "varlen_bf16_prefill_layer": PrefillLayerSpec("varlen_bf16_prefill_layer", io="bf16", h_qk=16,
                                                  h_v=16, seed=1016, varlen_range=(512, 8192),
                                                  n_varlen=8),
}


def any_workload(name: str):
    """Draw any named workload: the scan's, the convolution's or the norm's."""
    if name in WORKLOADS:
        return draw(WORKLOADS[name])
    if name in PREFILL_NORM_WORKLOADS:
        return draw_prefill_norm(PREFILL_NORM_WORKLOADS[name])
    if name in CONV_WORKLOADS:
        return draw_conv(CONV_WORKLOADS[name])
    if name in LAYER_WORKLOADS:
        return draw_layer(LAYER_WORKLOADS[name])
    if name in PREFILL_LAYER_WORKLOADS:
        return draw_prefill_layer(PREFILL_LAYER_WORKLOADS[name])
    return draw_norm(NORM_WORKLOADS[name])


ALL_WORKLOADS = sorted(list(WORKLOADS) + list(CONV_WORKLOADS) + list(NORM_WORKLOADS) +
                       list(LAYER_WORKLOADS) + list(PREFILL_NORM_WORKLOADS) +
                       list(PREFILL_LAYER_WORKLOADS))
