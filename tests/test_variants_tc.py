"""GPU parity of gdn_prefill_variant -- the update rules (gated_delta, delta, gated, linear),
one beta shared by every head and one decay per key dimension on the chunked tensor-core
prefill (16-bit I/O, d_k = d_v = 128) -- against the CPU oracle run on the same drawn
inputs.  The shapes cover ragged chunk tails, packed sequences (one of a single token),
GQA, an initial state and the time-parallel scan; per-key decay also runs with decay
strong enough that most in-chunk factors underflow, and with too small a workspace (the
token-sequential kernel).  Tolerances as in test_parity."""
import dataclasses

import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err, to_device

RULES = ("gated_delta", "delta", "gated", "linear")


def _stronger_decay(inp, by=3.0):
    """The same draw with A_log raised by `by` on every other key dimension, so that those
    dimensions decay e^by times faster (about -20 to -160 per token)."""
    bump = torch.zeros_like(inp.A_log)
    bump[..., 1::2] = by
    A_log = (inp.A_log + bump).to(torch.float32)
    f64 = dict(inp.f64)
    f64["A_log"] = A_log.to(torch.float64).numpy().reshape(-1)
    return dataclasses.replace(inp, A_log=A_log, f64=f64)


def _run(inp, rule, workspace=None):
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_prefill_variant
    s = inp.spec
    d = to_device(inp)
    o, state = gdn_prefill_variant(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                   d["dt_bias"], d["state_in"], d["cu_seqlens"], inp.scale,
                                   rule=rule, decay_per_key=s.decay_per_key,
                                   beta_shared=s.beta_shared, workspace=workspace)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    return o.float().cpu().numpy().reshape(-1, s.h_v, s.d_v), state.cpu().numpy()


def _check(inp, rule, what):
    o, s = _run(inp, rule)
    o_ref, s_ref = oracle.scan_inputs(inp, rule=rule, threads=8)
    tol = TOL[inp.spec.io]
    eo, es = rel_err(o, o_ref), rel_err(s, s_ref)
    print(f"{what} {rule}: o {eo:.3e}, state {es:.3e}")
    assert eo <= tol and es <= tol


def _tc_path(inp):
    from recurrent_state_scan_gb300 import gdn
    shape = gdn.shape_of_spec(inp.spec, inp.n_seq, inp.total_tokens)
    return gdn.gdn_prefill_variant_plan(shape, inp.spec.rule, inp.spec.decay_per_key,
                                        inp.spec.beta_shared)[0]


@pytest.mark.gpu
@pytest.mark.parametrize("rule", RULES)
def test_rules_on_the_tensor_core_prefill_batched(rule):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=300, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=311))
    assert _tc_path(inp) in (gdn.PATH_TC, gdn.PATH_TC_TP)
    _check(inp, rule, "batched")


@pytest.mark.gpu
@pytest.mark.parametrize("rule", RULES)
def test_rules_on_the_tensor_core_prefill_packed(rule):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.draw(workloads.small_spec(io="f16", lengths=(1, 129, 64, 250), h_qk=1, h_v=2,
                                              d_k=128, d_v=128, state_std=0.05, seed=312))
    _check(inp, rule, "packed")


@pytest.mark.gpu
@pytest.mark.parametrize("rule", ["gated_delta", "delta"])
def test_shared_beta_on_the_tensor_core_prefill(rule):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=3, seqlen=200, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=313,
                                              beta_shared=True))
    _check(inp, rule, "shared beta")


@pytest.mark.gpu
@pytest.mark.parametrize("rule", ["delta", "linear"])
def test_rules_on_the_time_parallel_scan(rule):
    """A single 2,048-token sequence at 4 value heads: 8 chains, so the scan is cut into
    segments scanned at once and combined."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=1, seqlen=2048, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=314))
    assert _tc_path(inp) == gdn.PATH_TC_TP
    _check(inp, rule, "time-parallel")


@pytest.mark.gpu
@pytest.mark.parametrize("rule", ["gated_delta", "gated"])
def test_per_key_decay_on_the_tensor_core_prefill_batched(rule):
    """Two 300-token sequences (a ragged last chunk), GQA 2 -> 4 heads, an initial state."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=300, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=315,
                                              decay_per_key=True))
    assert _tc_path(inp) in (gdn.PATH_TC, gdn.PATH_TC_TP)
    _check(inp, rule, "per-key batched")


@pytest.mark.gpu
@pytest.mark.parametrize("rule", ["gated_delta", "gated"])
def test_per_key_decay_on_the_tensor_core_prefill_packed(rule):
    """Packed f16 sequences of 1, 129, 64 and 250 tokens: a ragged chunk's padded rows
    belong to the next sequence, and its Q~ / K~ rows are not overwritten."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.draw(workloads.small_spec(io="f16", lengths=(1, 129, 64, 250), h_qk=1, h_v=2,
                                              d_k=128, d_v=128, state_std=0.05, seed=316,
                                              decay_per_key=True))
    _check(inp, rule, "per-key packed")


@pytest.mark.gpu
def test_per_key_decay_on_the_time_parallel_scan():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=1, seqlen=2048, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=317,
                                              decay_per_key=True))
    assert _tc_path(inp) == gdn.PATH_TC_TP
    _check(inp, "gated_delta", "per-key time-parallel")


@pytest.mark.gpu
@pytest.mark.parametrize("io", ["bf16", "f16"])
def test_per_key_decay_strong(io):
    """Half the key dimensions decay by up to ~160 per token: most e^{G_t - G_s} inside a
    chunk underflow, none may overflow."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = _stronger_decay(workloads.draw(workloads.small_spec(
        io=io, lengths=(200, 77, 300), h_qk=2, h_v=2, d_k=128, d_v=128, state_std=0.05,
        seed=318, decay_per_key=True)))
    _check(inp, "gated_delta", "per-key strong decay")


@pytest.mark.gpu
def test_per_key_decay_with_the_records_only_workspace():
    """With gdn_prefill_workspace_bytes (no room for Q~ and K~) the call runs the
    token-sequential kernel: same results."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=130, h_qk=2, h_v=2,
                                              d_k=128, d_v=128, state_std=0.05, seed=319,
                                              decay_per_key=True))
    shape = gdn.shape_of_spec(inp.spec, inp.n_seq, inp.total_tokens)
    small = gdn.gdn_prefill_workspace_bytes(shape)
    assert gdn.gdn_prefill_variant_workspace_bytes(shape, "gated_delta", True) > small
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    o, s = _run(inp, "gated_delta", workspace=ws)
    o_ref, s_ref = oracle.scan_inputs(inp, rule="gated_delta", threads=8)
    tol = TOL[inp.spec.io]
    assert rel_err(o, o_ref) <= tol and rel_err(s, s_ref) <= tol


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["bf16_delta_prefill_t4096", "bf16_shared_beta_prefill_t4096",
                                  "bf16_perkey_prefill_t4096"])
def test_full_size_variant_workloads(name):
    """The measured prefill-length variants, every element against the oracle, all on the
    tensor-core path (time-parallel at this shape)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.workload(name)
    _check(inp, inp.spec.rule, name)


@pytest.mark.gpu
def test_per_key_decay_with_a_off_16_bytes():
    """The per-key prep loads a's tiles by TMA; an `a` 2 bytes past a 16-byte boundary takes
    the token-sequential kernel instead, with the same results."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_prefill_variant
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=130, h_qk=2, h_v=2,
                                              d_k=128, d_v=128, state_std=0.05, seed=320,
                                              decay_per_key=True))
    d = to_device(inp)
    buf = torch.empty(d["a"].numel() + 1, dtype=d["a"].dtype, device="cuda")
    a_off = buf[1:].view(d["a"].shape)
    a_off.copy_(d["a"])
    o, st = gdn_prefill_variant(d["q"], d["k"], d["v"], a_off, d["b"], d["A_log"], d["dt_bias"],
                                d["state_in"], d["cu_seqlens"], inp.scale, decay_per_key=True)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    o_ref, s_ref = oracle.scan_inputs(inp, threads=8)
    tol = TOL[inp.spec.io]
    assert rel_err(o.float().cpu().numpy().reshape(-1, 2, 128), o_ref) <= tol
    assert rel_err(st.cpu().numpy(), s_ref) <= tol
