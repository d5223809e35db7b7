"""GPU parity of gdn_prefill_layer -- the causal conv (onnxruntime-ep-mlx ssm.rs
`causal_conv_op`), as a streaming pass before the prefill (fuse = 0) or inside the chunked
prefill's prep (fuse = 1), the prefill (the CUDA page's `linear_attention_core` Steps 1-4)
and the gated RMS norm (ssm.rs `gated_rms_norm_op`).  Both forms are checked.

References:
  * the float64 oracle chain: the oracle's convolution per sequence, its output rounded
    to the I/O type (as a stored conv output would be), split into q, k and v; the
    oracle's scan; o rounded to the I/O type; the oracle's gated RMS norm.  y and the
    state are held to the scan's tolerance (max|d| / max|ref|); the present conv state is
    a copy of inputs and must match exactly;
  * for batched inputs, the separate GPU calls gdn_causal_conv -> gdn_prefill ->
    gdn_gated_rmsnorm on the same inputs: the fused form convolves in the same fp32 order,
    so y may differ only through the scan's and the norm's sums -- within one rounding
    step of the I/O type, element by element -- and the conv state is bit for bit the same.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}
ULP = {"bf16": 2.0 ** -7, "f16": 2.0 ** -10}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _io(x, io):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DT[io]).double().numpy()


def _oracle(inp, with_state=True):
    s, f, cu = inp.spec, inp.f64, inp.cu_seqlens
    C = 2 * s.h_qk * 128 + s.h_v * 128
    K, N = s.kernel, inp.n_seq
    x = f["x"].reshape(-1, C)
    st = f["conv_state"] if with_state else np.zeros((N, K - 1, C))
    yc = np.zeros_like(x)
    cs = np.zeros((N, K - 1, C))
    for n in range(N):
        a0, a1 = int(cu[n]), int(cu[n + 1])
        if a1 == a0:
            cs[n] = st[n]
            continue
        y1, s1 = oracle.causal_conv(x[a0:a1][None], f["w"], f["bias"], st[n][None], silu=s.silu)
        yc[a0:a1], cs[n] = y1[0], s1[0]
    yc = _io(yc, s.io)
    q, k, v = yc[:, :s.h_qk * 128], yc[:, s.h_qk * 128:2 * s.h_qk * 128], yc[:, 2 * s.h_qk * 128:]
    o, state = oracle.scan(cu, s.h_qk, s.h_v, 128, 128, q, k, v, a=f["a"], b=f["b"], A_log=f["A_log"],
                           dt_bias=f["dt_bias"], state_in=f["state_in"], scale=inp.scale, threads=8)
    y = oracle.gated_rmsnorm(_io(o, s.io).reshape(-1, 128), f["norm_scale"], f["gate"].reshape(-1, 128),
                             s.eps, s.activation)
    return y.reshape(-1, s.h_v, 128), state, cs


def _fused(inp, with_state=True, bias=True, fuse=False):
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_prefill_layer
    s = inp.spec
    d = lambda t: None if t is None else t.cuda()
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda") if inp.varlen else None
    y, st, cs = gdn_prefill_layer(d(inp.x), d(inp.w), d(inp.bias) if bias else None,
                                  d(inp.conv_state) if with_state else None, d(inp.a), d(inp.b),
                                  d(inp.A_log), d(inp.dt_bias), d(inp.state_in), cu, d(inp.norm_scale),
                                  d(inp.gate), h_qk=s.h_qk, h_v=s.h_v, scale=inp.scale,
                                  conv_activation="silu" if s.silu else "none",
                                  norm_activation=s.activation, eps=s.eps, fuse=fuse)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    return y, st, cs


def _against_oracle(inp, with_state=True, fuse=False):
    s = inp.spec
    y, st, cs = _fused(inp, with_state, bias=inp.bias is not None, fuse=fuse)
    y_ref, s_ref, cs_ref = _oracle(inp, with_state)
    ey = rel_err(y.float().cpu().numpy().reshape(-1, s.h_v, 128), y_ref)
    es = rel_err(st.cpu().numpy(), s_ref)
    print(f"y {ey:.3e}, state {es:.3e}")
    assert ey <= TOL[s.io] and es <= TOL[s.io]
    assert np.array_equal(cs.double().cpu().numpy(), _io(cs_ref, s.io))


def _spec(**kw):
    base = dict(name="t", io="bf16", h_qk=2, h_v=4, seed=701)
    base.update(kw)
    return workloads.PrefillLayerSpec(**base)


@pytest.mark.parametrize("fuse", [False, True])
def test_batched_gqa_ragged_against_the_oracle_chain(fuse):
    """Two 300-token sequences (a ragged last chunk), GQA 2 -> 4 heads, a conv bias and
    state, an initial state."""
    _against_oracle(workloads.draw_prefill_layer(_spec(batch=2, seqlen=300)), fuse=fuse)


@pytest.mark.parametrize("fuse", [False, True])
def test_packed_short_and_empty_sequences_against_the_oracle_chain(fuse):
    """Packed sequences of 1, 2, 0, 129, 64 and 250 tokens: the first two are shorter than
    the conv window (their present state mixes the past state and their inputs), one is
    empty (its state passes through), and chunk tails hold the next sequence's rows."""
    _against_oracle(workloads.draw_prefill_layer(_spec(io="f16", lengths=(1, 2, 0, 129, 64, 250),
                                                       h_qk=1, h_v=2, seed=702)), fuse=fuse)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("K", [1, 2, 3])
def test_fewer_taps_no_bias_no_state_no_activation(K, fuse):
    # Without silu the convolved keys are twice as large: x_std 0.12 keeps |k|^2 below 1.
    inp = workloads.draw_prefill_layer(_spec(batch=1, seqlen=200, kernel=K, bias=False, silu=False,
                                             x_std=0.12, h_qk=1, h_v=2, seed=703 + K))
    _against_oracle(inp, with_state=False, fuse=fuse)


def test_time_parallel_shape_against_the_oracle_chain():
    """One 2,048-token sequence at 4 value heads: the scan runs time-parallel."""
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw_prefill_layer(_spec(batch=1, seqlen=2048, h_qk=2, h_v=4, seed=707))
    shape = gdn.make_shape(gdn.GDN_BF16, 1, 2048, 1, 2, 4, 128, 128)
    assert gdn.gdn_prefill_plan(shape)[0] == gdn.PATH_TC_TP
    _against_oracle(inp)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("io", ["bf16", "f16"])
def test_equals_the_separate_calls(io, fuse):
    """Batched: gdn_causal_conv -> gdn_prefill -> gdn_gated_rmsnorm on the same inputs."""
    from recurrent_state_scan_gb300 import (gdn_causal_conv, gdn_gated_rmsnorm, gdn_last_device_status,
                                            gdn_prefill)
    inp = workloads.draw_prefill_layer(_spec(io=io, batch=3, seqlen=333, seed=708))
    s = inp.spec
    y, st, cs = _fused(inp, fuse=fuse)
    x = inp.x.cuda()
    yc, cs2 = gdn_causal_conv(x, inp.w.cuda(), inp.bias.cuda(), inp.conv_state.cuda(), activation="silu")
    B, T = x.shape[0], x.shape[1]
    q = yc[..., :s.h_qk * 128].contiguous().view(B, T, s.h_qk, 128)
    k = yc[..., s.h_qk * 128:2 * s.h_qk * 128].contiguous().view(B, T, s.h_qk, 128)
    v = yc[..., 2 * s.h_qk * 128:].contiguous().view(B, T, s.h_v, 128)
    o, st2 = gdn_prefill(q, k, v, inp.a.cuda(), inp.b.cuda(), inp.A_log.cuda(), inp.dt_bias.cuda(),
                         inp.state_in.cuda(), None, inp.scale)
    y2 = gdn_gated_rmsnorm(o, inp.norm_scale.cuda(), inp.gate.cuda(), s.eps, s.activation)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    assert torch.equal(cs, cs2)
    assert torch.equal(st, st2)
    a_, b_ = y.double().cpu().numpy(), y2.double().cpu().numpy()
    bound = ULP[io] * np.abs(b_) + 1e-6 * np.max(np.abs(b_))
    assert not (np.abs(a_ - b_) > bound).any()


@pytest.mark.parametrize("fuse", [False, True])
def test_full_size_layer_workload_against_the_oracle_chain(fuse):
    _against_oracle(workloads.any_workload("varlen_bf16_prefill_layer"), fuse=fuse)


def test_bad_arguments_are_rejected():
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw_prefill_layer(_spec(batch=1, seqlen=64, h_qk=1, h_v=1, seed=709))
    d = lambda t: t.cuda()
    args = [d(inp.x), d(inp.w), d(inp.bias), d(inp.conv_state), d(inp.a), d(inp.b), d(inp.A_log),
            d(inp.dt_bias), None, None, d(inp.norm_scale), d(inp.gate)]
    with pytest.raises(gdn.GdnError):      # the conv state updated in place
        gdn.gdn_prefill_layer(*args, h_qk=1, h_v=1, conv_state_out=args[3])
    w5 = torch.zeros((inp.w.shape[0], 1, 5), dtype=inp.w.dtype, device="cuda")
    with pytest.raises(gdn.GdnError):      # five taps
        gdn.gdn_prefill_layer(args[0], w5, *args[2:], h_qk=1, h_v=1)
