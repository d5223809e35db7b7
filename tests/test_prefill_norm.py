"""GPU parity of gdn_prefill_norm -- the prefill followed by the gated RMS norm of its output
over each d_v row (the CUDA page's linear_attention_core Steps 1-4, then the
onnxruntime-ep-mlx ssm.rs page's GatedRMSNorm).  By default the norm is a second launch,
in place on y; with fuse=True, on the chunked tensor-core path, it runs in the scan
(the two column halves of a head as a cluster pair, the state warps norming each staged
tile one chunk behind the readout).  Both forms are checked.

References:
  * the float64 oracle chain: the oracle's scan, its o rounded to the I/O type (the GPU
    rounds o there too, as a stored o would be), then the oracle's gated RMS norm.  y is
    held to the scan's tolerance (TOL, max|d| / max|ref|), the state likewise;
  * the separate GPU calls, gdn_prefill then gdn_gated_rmsnorm: the same o values, so y may
    differ only through the order of a row's sum of squares -- at most one rounding step
    of the I/O type, checked element by element -- and the state is bit for bit the same.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

ULP = {"bf16": 2.0 ** -7, "f16": 2.0 ** -10, "f32": 1e-6}
DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _norm_inputs(inp, activation, seed):
    """norm_scale [d_v] and gate (o's shape), drawn by the shared seeded generator."""
    s = inp.spec
    shape = (inp.total_tokens, s.h_v, s.d_v)
    n = workloads.draw_norm(workloads.NormSpec("t", s.io, shape, seed, eps=1e-6,
                                               activation=activation))
    return n.scale, n.gate, n.spec.eps


def _fused(inp, scale, gate, eps, activation, gate_offset=0, fuse=True):
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_prefill_norm
    d = to_device(inp)
    g = gate.cuda().view(d["v"].shape)
    if gate_offset:
        buf = torch.empty(g.numel() + gate_offset, dtype=g.dtype, device="cuda")
        g2 = buf[gate_offset:].view(g.shape)
        g2.copy_(g)
        g = g2
    shape_o = d["v"].shape
    y, st = gdn_prefill_norm(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                             d["state_in"], d["cu_seqlens"], inp.scale, norm_scale=scale.cuda(),
                             gate=g, eps=eps, activation=activation, fuse=fuse)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    assert y.shape == shape_o
    return y, st


def _separate(inp, scale, gate, eps, activation):
    from recurrent_state_scan_gb300 import gdn_gated_rmsnorm, gdn_last_device_status, gdn_prefill
    d = to_device(inp)
    o, st = gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                        d["state_in"], d["cu_seqlens"], inp.scale)
    y = gdn_gated_rmsnorm(o, scale.cuda(), gate.cuda().view(o.shape), eps, activation)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    return y, st


def _oracle(inp, scale, gate, eps, activation):
    s = inp.spec
    o_ref, s_ref = oracle.scan_inputs(inp, threads=8)
    o_io = torch.from_numpy(np.ascontiguousarray(o_ref)).to(DT[s.io]).double().numpy()
    y_ref = oracle.gated_rmsnorm(o_io.reshape(-1, s.d_v), scale.double().numpy(),
                                 gate.double().numpy().reshape(-1, s.d_v), eps, activation)
    return y_ref.reshape(-1, s.h_v, s.d_v), s_ref


def _against_oracle(inp, activation, seed, fuse=True):
    s = inp.spec
    scale, gate, eps = _norm_inputs(inp, activation, seed)
    y, st = _fused(inp, scale, gate, eps, activation, fuse=fuse)
    y_ref, s_ref = _oracle(inp, scale, gate, eps, activation)
    ey = rel_err(y.float().cpu().numpy().reshape(-1, s.h_v, s.d_v), y_ref)
    es = rel_err(st.cpu().numpy(), s_ref)
    print(f"y {ey:.3e}, state {es:.3e}")
    assert ey <= TOL[s.io] and es <= TOL[s.io]


def _against_separate(inp, activation, seed, gate_offset=0, fuse=True):
    s = inp.spec
    scale, gate, eps = _norm_inputs(inp, activation, seed)
    y, st = _fused(inp, scale, gate, eps, activation, gate_offset, fuse=fuse)
    y2, st2 = _separate(inp, scale, gate, eps, activation)
    a = y.double().cpu().numpy()
    b = y2.double().cpu().numpy()
    bound = ULP[s.io] * np.abs(b) + 1e-6 * np.max(np.abs(b))
    bad = np.abs(a - b) > bound
    assert not bad.any(), f"{bad.sum()} of {a.size} elements differ by more than one rounding"
    assert torch.equal(st, st2)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("io", ["bf16", "f16"])
@pytest.mark.parametrize("activation", ["silu", "sigmoid"])
def test_batched_against_the_oracle_chain(io, activation, fuse):
    """Two 300-token sequences (a ragged last chunk), GQA 2 -> 4 heads, an initial state."""
    inp = workloads.draw(workloads.small_spec(io=io, batch=2, seqlen=300, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=501))
    _against_oracle(inp, activation, 601, fuse=fuse)


@pytest.mark.parametrize("fuse", [False, True])
def test_packed_against_the_oracle_chain(fuse):
    """Packed sequences of 1, 129, 64 and 250 tokens: rows of the next sequence share a
    chunk tile with a ragged last chunk, and are neither normed nor stored by it."""
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=(1, 129, 64, 250), h_qk=1,
                                              h_v=2, d_k=128, d_v=128, state_std=0.05,
                                              seed=502))
    _against_oracle(inp, "silu", 602, fuse=fuse)


@pytest.mark.parametrize("io", ["bf16", "f16"])
def test_equals_the_separate_calls(io):
    inp = workloads.draw(workloads.small_spec(io=io, lengths=(70, 300, 5, 192), h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=503))
    _against_separate(inp, "silu", 603)


def test_gate_off_16_bytes_takes_the_second_launch():
    """fuse=True with a gate 8 bytes past a 16-byte boundary: the tensor-core prefill
    writes o into y and the norm runs after it, in place; same values as the separate
    calls."""
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=200, h_qk=2, h_v=2,
                                              d_k=128, d_v=128, state_std=0.05, seed=504))
    _against_separate(inp, "sigmoid", 604, gate_offset=4)


@pytest.mark.parametrize("io,d_k", [("f32", 128), ("bf16", 64)])
def test_off_the_tensor_core_path(io, d_k):
    """f32 I/O or d_k = 64: the token-sequential scan, then the norm as a second launch."""
    inp = workloads.draw(workloads.small_spec(io=io, batch=2, seqlen=40, h_qk=2, h_v=2,
                                              d_k=d_k, d_v=64, state_std=0.05, seed=505))
    _against_oracle(inp, "silu", 605)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("name", ["varlen_bf16_prefill", "gqa_f16_prefill"])
def test_full_size_against_the_separate_calls(name, fuse):
    """Every element of the full-size packed and GQA workloads (32K and 16K tokens)."""
    inp = workloads.workload(name)
    _against_separate(inp, "silu", 606, fuse=fuse)


def test_full_size_varlen_against_the_oracle_chain():
    inp = workloads.workload("varlen_bf16_prefill")
    _against_oracle(inp, "silu", 607)


def test_y_overlapping_the_gate_is_rejected():
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=1, seqlen=64, h_qk=1, h_v=1,
                                              d_k=128, d_v=128, seed=506))
    scale, gate, eps = _norm_inputs(inp, "silu", 606)
    d = to_device(inp)
    g = gate.cuda().view(d["v"].shape)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_norm(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                             None, None, inp.scale, norm_scale=scale.cuda(), gate=g, y=g)
