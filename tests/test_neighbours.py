"""GPU parity of the layer ops around the scan -- the causal depthwise convolution with a
carried state (gdn_causal_conv, gdn_causal_conv_slots) and the gated RMS norm
(gdn_gated_rmsnorm) -- with the float64 CPU oracle on the same drawn inputs.

Tolerance, from the arithmetic: the GPU evaluates in fp32 and rounds each output once
to the I/O dtype, so an output may differ from the exact value by half an ulp of the
I/O dtype (relative 2^-9 for bf16, 2^-12 for f16) plus fp32 evaluation error, which is
bounded by a few fp32 ulps of the largest term.  The check is element by element:
|gpu - ref| <= rel * |ref| + 1e-5 * max|ref|, rel = 2^-8 (bf16), 2^-11 (f16), 1e-5 (f32).
The present states are copies of inputs and must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

REL = {"f32": 1e-5, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _close(gpu, ref, io):
    gpu = gpu.double().cpu().numpy() if isinstance(gpu, torch.Tensor) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    if ref.size == 0:
        return
    bound = REL[io] * np.abs(ref) + 1e-5 * np.max(np.abs(ref))
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, worst " \
                          f"{np.max(np.abs(gpu - ref) - bound):.3g} over the bound"


def _exact(gpu, ref):
    assert np.array_equal(gpu.double().cpu().numpy(), np.asarray(ref, dtype=np.float64))


def _status_ok():
    from recurrent_state_scan_gb300 import gdn_last_device_status
    assert gdn_last_device_status() == 0


def _conv_case(io, B, L, C, K, dil, channels_last=True, silu=True, bias=True, state=True,
               window=0, seed=0):
    spec = workloads.ConvSpec("t", io, B, L, C, seed, kernel=K, dilation=dil,
                              channels_last=channels_last, silu=silu, bias=bias,
                              state_std=1.0 if state else 0.0, state_window=window)
    return workloads.draw_conv(spec)


def _run_conv(inp, in_place=False):
    from recurrent_state_scan_gb300 import gdn_causal_conv
    s = inp.spec
    dev = lambda t: None if t is None else t.cuda()
    x, w, b, st = dev(inp.x), dev(inp.w), dev(inp.bias), dev(inp.state_in)
    y, so = gdn_causal_conv(x, w, b, st, dilation=s.dilation, channels_last=s.channels_last,
                            activation="silu" if s.silu else "none",
                            state_window=s.state_window,
                            state_out=st if in_place else None)
    torch.cuda.synchronize()
    _status_ok()
    return y, so


def _conv_ref(inp):
    s, f = inp.spec, inp.f64
    return oracle.causal_conv(f["x"], f["w"], f["bias"], f["state_in"], dilation=s.dilation,
                              channels_last=s.channels_last, silu=s.silu,
                              state_window=s.state_window)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("geom", [
    # (C, K, dilation, channels_last, silu, bias)
    (24, 4, 1, True, True, True),      # four channels a thread, four taps in registers
    (24, 3, 1, True, False, True),
    (13, 4, 1, True, True, False),     # one channel a thread
    (24, 1, 1, True, True, True),      # no carry
    (24, 4, 2, True, True, True),      # dilated: taps through L1
    (8, 2, 9, True, False, False),     # carry 9
    (24, 5, 1, True, True, True),      # five taps
    (16, 4, 1, False, True, True),     # channels first
    (7, 3, 3, False, False, True),
])
def test_conv_matches_oracle(io, geom):
    C, K, dil, last, silu, bias = geom
    inp = _conv_case(io, 3, 37, C, K, dil, last, silu, bias, seed=K * 10 + dil)
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, io)
    _exact(so, s_ref)


@pytest.mark.parametrize("L", [0, 1, 2, 7, 8, 9, 16, 17, 63, 100])
def test_conv_lengths_around_the_tile(L):
    inp = _conv_case("bf16", 2, L, 32, 4, 1, seed=L)
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, "bf16")
    _exact(so, s_ref)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("L,C,K", [(64, 32, 4), (255, 264, 4), (256, 512, 3), (257, 40, 2),
                                   (600, 264, 1), (1000, 16, 4)])
def test_conv_long_rows_through_shared_memory(io, L, C, K):
    """Rows of 64 tokens or more stream through shared memory in 32-token stages and
    256-token chunks (partial channel slabs and ragged chunks included)."""
    inp = _conv_case(io, 2, L, C, K, 1, seed=L + C + K)
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, io)
    _exact(so, s_ref)


@pytest.mark.parametrize("io", ["bf16", "f16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("silu,bias,state", [(True, True, True), (False, False, False)])
def test_conv_long_rows_every_tap_count(io, K, silu, bias, state):
    """16-bit long rows run on the bulk-copy kernel, compiled per tap count and activation.
    Without a past state a row's first stage has zero-filled rows; 520 channels leave an
    8-channel slab; 333 tokens end in a ragged stage of a ragged chunk."""
    inp = _conv_case(io, 2, 333, 520, K, 1, silu=silu, bias=bias, state=state,
                     seed=700 + 10 * K + int(silu))
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, io)
    _exact(so, s_ref)


def test_conv_long_rows_with_an_output_off_16_bytes():
    """y 8 bytes past a 16-byte boundary: the 8-byte-store staged kernel takes the call and
    gives the same values."""
    from recurrent_state_scan_gb300 import gdn_causal_conv
    inp = _conv_case("bf16", 2, 300, 64, 4, 1, seed=9)
    x, w, b, st = inp.x.cuda(), inp.w.cuda(), inp.bias.cuda(), inp.state_in.cuda()
    buf = torch.empty(x.numel() + 4, dtype=x.dtype, device="cuda")
    y = buf[4:].view(x.shape)
    assert y.data_ptr() % 16 == 8
    gdn_causal_conv(x, w, b, st, activation="silu", y=y)
    torch.cuda.synchronize()
    _status_ok()
    y_ref, _ = _conv_ref(inp)
    _close(y, y_ref, "bf16")
    y16, _ = gdn_causal_conv(x, w, b, st, activation="silu")
    torch.cuda.synchronize()
    assert torch.equal(y16, y)


def test_conv_long_rows_in_place():
    inp = _conv_case("bf16", 3, 300, 48, 4, 1, seed=8)
    y_ref, s_ref = _conv_ref(inp)
    y, so = _run_conv(inp, in_place=True)
    _close(y, y_ref, "bf16")
    _exact(so, s_ref)


@pytest.mark.parametrize("io", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("K,bias,state", [(4, True, True), (3, False, True), (2, True, False),
                                          (1, True, True), (4, False, False)])
def test_conv_decode_step(io, K, bias, state):
    """One token per row (the streaming decode kernel for 16-bit I/O), in place."""
    inp = _conv_case(io, 5, 1, 1032, K, 1, bias=bias, state=state, seed=500 + K)
    y_ref, s_ref = _conv_ref(inp)
    y, so = _run_conv(inp, in_place=state)
    _close(y, y_ref, io)
    _exact(so, s_ref)


def test_conv_without_past_state_starts_from_zeros():
    inp = _conv_case("bf16", 2, 9, 32, 4, 1, state=False, seed=5)
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, "bf16")
    _exact(so, s_ref)


@pytest.mark.parametrize("L", [0, 1, 2, 37])
@pytest.mark.parametrize("window", [1, 4, 8])
def test_conv_state_window(L, window):
    inp = _conv_case("bf16", 2, L, 24, 4, 1, window=window, seed=100 + L + window)
    y, so = _run_conv(inp)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, "bf16")
    _exact(so, s_ref)


@pytest.mark.parametrize("L,dil", [(1, 1), (37, 1), (2, 3), (37, 3)])
def test_conv_in_place_state(L, dil):
    inp = _conv_case("f16", 3, L, 24, 4, dil, seed=200 + L)
    y_ref, s_ref = _conv_ref(inp)
    y, so = _run_conv(inp, in_place=True)
    _close(y, y_ref, "f16")
    _exact(so, s_ref)


def test_conv_in_place_window():
    inp = _conv_case("bf16", 2, 3, 24, 4, 1, window=4, seed=300)
    y_ref, s_ref = _conv_ref(inp)
    y, so = _run_conv(inp, in_place=True)
    _close(y, y_ref, "bf16")
    _exact(so, s_ref)


def _slot_case(io, B, L, C, P, seed):
    spec = workloads.ConvSpec("t", io, B, L, C, seed, state_std=1.0, pool_size=P, bias=True)
    return workloads.draw_conv(spec)


@pytest.mark.parametrize("L", [1, 5, 130])
def test_conv_slots_match_oracle(L):
    from recurrent_state_scan_gb300 import gdn_causal_conv_slots
    inp = _slot_case("bf16", 6, L, 32, 16, seed=400 + L)
    pool = inp.pool.cuda()
    y = gdn_causal_conv_slots(inp.x.cuda(), inp.w.cuda(), pool, inp.slots.cuda(),
                              inp.bias.cuda(), activation="silu")
    torch.cuda.synchronize()
    _status_ok()
    f = inp.f64
    y_ref, p_ref = oracle.conv_slots(f["x"], f["w"], f["pool"], inp.slots.numpy(), f["bias"],
                                     silu=True)
    _close(y, y_ref, "bf16")
    _exact(pool, p_ref)


def test_conv_slot_outside_the_pool_skips_its_row():
    from recurrent_state_scan_gb300 import gdn_causal_conv_slots, gdn_last_device_status
    inp = _slot_case("bf16", 4, 3, 32, 8, seed=410)
    slots = inp.slots.clone()
    slots[2] = 8
    pool = inp.pool.cuda()
    y = torch.full(inp.x.shape, 7.0, dtype=torch.bfloat16, device="cuda")
    gdn_causal_conv_slots(inp.x.cuda(), inp.w.cuda(), pool, slots.cuda(), inp.bias.cuda(),
                          activation="silu", y=y)
    torch.cuda.synchronize()
    assert gdn_last_device_status() != 0
    f = inp.f64
    y_ref, p_ref = oracle.conv_slots(f["x"], f["w"], f["pool"], slots.numpy(), f["bias"],
                                     silu=True)
    _exact(pool, p_ref)
    assert torch.all(y[2] == 7.0)
    keep = [0, 1, 3]
    _close(y[keep], y_ref[keep], "bf16")


@pytest.mark.parametrize("name", sorted(workloads.CONV_WORKLOADS))
def test_conv_full_size_workloads(name):
    inp = workloads.any_workload(name)
    y, so = _run_conv(inp, in_place=inp.spec.decode)
    y_ref, s_ref = _conv_ref(inp)
    _close(y, y_ref, inp.spec.io)
    _exact(so, s_ref)


# ------------------------------------------------------------------ gated RMS norm

def _norm_case(io, shape, activation="silu", eps=1e-6, seed=0):
    return workloads.draw_norm(workloads.NormSpec("t", io, tuple(shape), seed, eps=eps,
                                                  activation=activation))


def _run_norm(inp, in_place=False):
    from recurrent_state_scan_gb300 import gdn_gated_rmsnorm
    s = inp.spec
    x = inp.x.cuda()
    y = gdn_gated_rmsnorm(x, inp.scale.cuda(), inp.gate.cuda(), s.eps, s.activation,
                          y=x if in_place else None)
    torch.cuda.synchronize()
    return y


def _norm_ref(inp):
    s, f = inp.spec, inp.f64
    return oracle.gated_rmsnorm(f["x"], f["scale"], f["gate"], s.eps, s.activation)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("width", [128, 64, 96, 30, 4096])
@pytest.mark.parametrize("activation", ["silu", "sigmoid"])
def test_norm_matches_oracle(io, width, activation):
    inp = _norm_case(io, (3, 13, width), activation, seed=width)
    _close(_run_norm(inp), _norm_ref(inp), io)


def test_norm_rows_of_128_off_16_bytes():
    """16-bit rows of 128 take the half-warp kernel when every pointer is 16-byte aligned;
    x and y 8 bytes off that boundary take the four-rows-a-warp kernel, same values."""
    from recurrent_state_scan_gb300 import gdn_gated_rmsnorm
    inp = _norm_case("bf16", (7, 9, 128), seed=11)
    ref = _norm_ref(inp)
    x = inp.x.cuda()
    buf = torch.empty(x.numel() + 4, dtype=x.dtype, device="cuda")
    xo = buf[4:].view(x.shape)
    xo.copy_(x)
    assert xo.data_ptr() % 16 == 8
    y = gdn_gated_rmsnorm(xo, inp.scale.cuda(), inp.gate.cuda(), inp.spec.eps, "silu")
    y16 = gdn_gated_rmsnorm(x, inp.scale.cuda(), inp.gate.cuda(), inp.spec.eps, "silu")
    torch.cuda.synchronize()
    _close(y, ref, "bf16")
    _close(y16, ref, "bf16")


def test_norm_in_place_and_eps():
    inp = _norm_case("bf16", (5, 4, 128), eps=0.5, seed=9)
    ref = _norm_ref(inp)
    _close(_run_norm(inp, in_place=True), ref, "bf16")


def test_norm_full_size_workload():
    inp = workloads.any_workload("bf16_norm_gqa")
    _close(_run_norm(inp), _norm_ref(inp), "bf16")
