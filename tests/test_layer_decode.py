"""gdn_decode_layer: one decode token of the layer (causal conv -> gated delta-rule step ->
gated RMS norm) in one launch.

The reference is the oracle's chain of the three ops, each pinned on its own elsewhere:
oracle.causal_conv (onnxruntime-ep-mlx ssm.rs `causal_conv_op`), oracle.scan for the one
token (onnx-runtime-ep-cuda linear_attention.rs `linear_attention_core`, Steps 1-4) and
oracle.gated_rmsnorm (ssm.rs `gated_rms_norm_op`), with q, k, v cut from the conv's
channels in the order [q | k | v].  The GPU tests compare y, the recurrent state and the
conv state element by element, over two tokens in a row (the conv states alternate
between two buffers), and also against the three separate library calls.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err


def oracle_layer(spec, f, conv_state, state):
    """The chain in float64: conv (silu) -> cut q, k, v -> one scan token -> gated norm."""
    B, dqk = spec.batch, spec.h_qk * 128
    yc, cs_out = oracle.causal_conv(f["x"], f["w"], f["bias"], conv_state, silu=True)
    q = yc[:, 0, :dqk].reshape(B, spec.h_qk, 128)
    k = yc[:, 0, dqk:2 * dqk].reshape(B, spec.h_qk, 128)
    v = yc[:, 0, 2 * dqk:].reshape(B, spec.h_v, spec.d_v)
    o, s_out = oracle.scan(np.arange(B + 1), spec.h_qk, spec.h_v, 128, spec.d_v, q, k, v,
                           a=f["a"].reshape(B, spec.h_v), b=f["b"].reshape(B, spec.h_v),
                           A_log=f["A_log"], dt_bias=f["dt_bias"], state_in=state,
                           threads=os.cpu_count() or 1)
    y = oracle.gated_rmsnorm(o.reshape(B, 1, spec.h_v, spec.d_v), f["norm_scale"], f["gate"],
                             eps=spec.eps, activation="silu")
    return y, s_out, cs_out


def _shape(gdn, io, batch, h_qk, h_v, d_k, d_v):
    return gdn.make_shape(io, batch, 1, batch, h_qk, h_v, d_k, d_v)


def test_layer_rejects_bad_arguments_on_the_host():
    from recurrent_state_scan_gb300 import gdn
    lib = gdn.load()
    P = 4096   # a 16-byte aligned address that is never dereferenced: the checks come first
    args = lambda cs_in, cs_out: ([ctypes.c_void_p(P)] * 3 + [ctypes.c_void_p(cs_in), ctypes.c_void_p(cs_out)]
                                  + [ctypes.c_void_p(P)] * 5 + [0.0] + [ctypes.c_void_p(P)] * 4)
    layer = gdn.GdnLayerParams(4, gdn.ACTIVATIONS["silu"], gdn.ACTIVATIONS["silu"], 1e-6)
    ok = _shape(gdn, gdn.GDN_BF16, 2, 1, 2, 128, 128)
    # The conv states may not overlap: several CTAs read the same q and k channels.
    st = lib.gdn_decode_layer(ctypes.byref(ok), ctypes.byref(layer), *args(P, P + 16))
    assert st == gdn.GDN_ERR_INVALID_ARG and b"overlaps" in lib.gdn_last_error_message()
    for bad_k in (0, 9):
        bad = gdn.GdnLayerParams(bad_k, 1, 1, 1e-6)
        assert lib.gdn_decode_layer(ctypes.byref(ok), ctypes.byref(bad), *args(P, P + (1 << 20))) == \
            gdn.GDN_ERR_INVALID_ARG
    bad_act = gdn.GdnLayerParams(4, gdn.ACTIVATIONS["silu"], gdn.ACTIVATIONS["none"], 1e-6)
    assert lib.gdn_decode_layer(ctypes.byref(ok), ctypes.byref(bad_act), *args(P, P + (1 << 20))) == \
        gdn.GDN_ERR_INVALID_ARG
    for d_k, d_v in ((64, 128), (128, 96)):
        sh = _shape(gdn, gdn.GDN_BF16, 2, 1, 2, d_k, d_v)
        assert lib.gdn_decode_layer(ctypes.byref(sh), ctypes.byref(layer), *args(P, P + (1 << 20))) == \
            gdn.GDN_ERR_UNSUPPORTED
    empty = _shape(gdn, gdn.GDN_BF16, 0, 1, 2, 128, 128)
    assert lib.gdn_decode_layer(ctypes.byref(empty), ctypes.byref(layer), *([None] * 10), 0.0,
                                *([None] * 4)) == gdn.GDN_OK


def test_oracle_chain_cuts_the_channels_in_order():
    """The chain reads q, k and v from consecutive channel blocks: with one-tap identity
    weights and no activation the conv passes x through, so q is x's first block."""
    spec = workloads.LayerSpec("t", io="f32", batch=1, h_qk=1, h_v=1, seed=7, kernel=1)
    f = workloads.draw_layer(spec).f64
    yc, _ = oracle.causal_conv(f["x"], np.ones((f["x"].shape[2], 1, 1)), None, None)
    assert np.array_equal(yc, f["x"])


CASES = [
    # io, batch, h_qk, h_v, d_v, K, bias, conv state drawn
    ("bf16", 3, 2, 4, 128, 4, False, True),
    ("f32", 2, 1, 2, 256, 3, True, True),
    ("f16", 2, 2, 2, 64, 1, False, False),
    ("bf16", 2, 1, 1, 128, 4, True, False),
]


@pytest.mark.gpu
@pytest.mark.parametrize("io,batch,h_qk,h_v,d_v,K,bias,with_state", CASES)
def test_layer_matches_the_oracle_chain_over_two_tokens(io, batch, h_qk, h_v, d_v, K, bias, with_state):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn_decode_layer, gdn_last_device_status
    spec = workloads.LayerSpec("t", io=io, batch=batch, h_qk=h_qk, h_v=h_v, seed=40 + K, d_v=d_v,
                               kernel=K, bias=bias)
    tok = [workloads.draw_layer(spec), workloads.draw_layer(dataclass_replace(spec, seed=90 + K))]
    dev = lambda t: None if t is None else t.cuda()
    first = tok[0]
    state = first.state.cuda().clone()
    ref_state = first.f64["state"]
    cs_in = first.conv_state.cuda().clone() if (with_state and K > 1) else None
    ref_cs = first.f64["conv_state"] if (with_state and K > 1) else None
    for step, inp in enumerate(tok):
        cs_out = torch.empty_like(first.conv_state).cuda() if K > 1 else None
        y = gdn_decode_layer(dev(inp.x), dev(inp.w), dev(inp.bias) if bias else None, cs_in, cs_out,
                             dev(inp.a), dev(inp.b), dev(first.A_log), dev(first.dt_bias), state,
                             dev(inp.norm_scale), dev(inp.gate), h_qk=h_qk, h_v=h_v, eps=spec.eps)
        torch.cuda.synchronize()
        assert gdn_last_device_status() == 0
        f = dict(inp.f64)
        f["A_log"], f["dt_bias"] = first.f64["A_log"], first.f64["dt_bias"]
        if not bias:
            f["bias"] = None
        y_ref, ref_state, cs_ref = oracle_layer(spec, f, ref_cs, ref_state)
        ey = rel_err(y.float().cpu().numpy(), y_ref)
        es = rel_err(state.cpu().numpy(), ref_state)
        print(f"{io} K={K} step {step}: y {ey:.3e}, state {es:.3e}")
        assert ey <= TOL[io] and es <= TOL[io]
        if K > 1:
            # The present conv state is a copy of inputs: exact.
            assert np.array_equal(cs_out.double().cpu().numpy(), cs_ref)
        cs_in, ref_cs = cs_out, (cs_ref if K > 1 else None)   # the next token reads it


def dataclass_replace(spec, **kw):
    import dataclasses
    return dataclasses.replace(spec, **kw)


@pytest.mark.gpu
def test_layer_matches_the_three_separate_calls():
    """The fused step equals gdn_causal_conv -> gdn_decode_step -> gdn_gated_rmsnorm up to
    the order of fp32 sums (and the conv's activation, one ulp of the I/O type)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import (gdn_causal_conv, gdn_decode_layer, gdn_decode_step,
                                            gdn_gated_rmsnorm)
    spec = workloads.LayerSpec("t", io="bf16", batch=8, h_qk=2, h_v=4, seed=77, bias=True)
    inp = workloads.draw_layer(spec)
    c = {n: getattr(inp, n).cuda() for n in ("x", "w", "bias", "conv_state", "a", "b", "A_log",
                                            "dt_bias", "state", "norm_scale", "gate")}
    B, dqk = spec.batch, spec.h_qk * 128
    s_fused = c["state"].clone()
    y_fused = gdn_decode_layer(c["x"], c["w"], c["bias"], c["conv_state"],
                               torch.empty_like(c["conv_state"]), c["a"], c["b"], c["A_log"],
                               c["dt_bias"], s_fused, c["norm_scale"], c["gate"], h_qk=spec.h_qk,
                               h_v=spec.h_v, eps=spec.eps)
    yc, _ = gdn_causal_conv(c["x"], c["w"], c["bias"], c["conv_state"], activation="silu")
    q = yc[:, :, :dqk].reshape(B, 1, spec.h_qk, 128).contiguous()
    k = yc[:, :, dqk:2 * dqk].reshape(B, 1, spec.h_qk, 128).contiguous()
    v = yc[:, :, 2 * dqk:].reshape(B, 1, spec.h_v, spec.d_v).contiguous()
    s_sep = c["state"].clone()
    o = gdn_decode_step(q, k, v, c["a"], c["b"], c["A_log"], c["dt_bias"], s_sep)
    y_sep = gdn_gated_rmsnorm(o, c["norm_scale"], c["gate"], eps=spec.eps)
    torch.cuda.synchronize()
    assert rel_err(y_fused.float().cpu().numpy(), y_sep.float().cpu().numpy()) <= 2e-2
    assert rel_err(s_fused.cpu().numpy(), s_sep.cpu().numpy()) <= 1e-2


@pytest.mark.gpu
def test_layer_full_size_against_the_oracle_chain():
    """The measured workload (B = 256, 32 heads, d = 128, 4 taps), every unit compared."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn_decode_layer
    inp = workloads.any_workload("bf16_layer_decode_b256")
    spec = inp.spec
    state = inp.state.cuda()
    cs_out = torch.empty_like(inp.conv_state).cuda()
    y = gdn_decode_layer(inp.x.cuda(), inp.w.cuda(), None, inp.conv_state.cuda(), cs_out,
                         inp.a.cuda(), inp.b.cuda(), inp.A_log.cuda(), inp.dt_bias.cuda(), state,
                         inp.norm_scale.cuda(), inp.gate.cuda(), h_qk=spec.h_qk, h_v=spec.h_v,
                         eps=spec.eps)
    torch.cuda.synchronize()
    y_ref, s_ref, cs_ref = oracle_layer(spec, inp.f64, inp.f64["conv_state"], inp.f64["state"])
    ey, es = rel_err(y.float().cpu().numpy(), y_ref), rel_err(state.cpu().numpy(), s_ref)
    print(f"bf16_layer_decode_b256: y {ey:.3e}, state {es:.3e}")
    assert ey <= TOL["bf16"] and es <= TOL["bf16"]
    assert np.array_equal(cs_out.double().cpu().numpy(), cs_ref)
