"""GPU parity of gdn_prefill_variant -- the update rules (gated_delta, delta, gated, linear)
and one beta shared by every head on the chunked tensor-core prefill (16-bit I/O,
d_k = d_v = 128), and per-key decay through the same entry point on the token-sequential
kernel -- against the CPU oracle run on the same drawn inputs.  The shapes cover ragged
chunk tails, packed sequences (one of a single token), GQA, an initial state and the
time-parallel scan.  Tolerances as in test_parity."""
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err, to_device

RULES = ("gated_delta", "delta", "gated", "linear")


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
    return gdn.gdn_prefill_plan(shape)[0]


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
def test_per_key_decay_through_the_prefill_entry_point():
    """Per-key decay is not on the tensor-core path: the same entry point runs it on the
    token-sequential kernel, with no workspace."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=2, seqlen=70, h_qk=2, h_v=4,
                                              d_k=128, d_v=128, state_std=0.05, seed=315,
                                              decay_per_key=True))
    _check(inp, "gated_delta", "per-key decay")


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["bf16_delta_prefill_t4096", "bf16_shared_beta_prefill_t4096",
                                  "bf16_perkey_prefill_t4096"])
def test_full_size_variant_workloads(name):
    """The measured prefill-length variants, every element against the oracle: the delta
    rule and the shared beta on the tensor-core path (time-parallel at this shape),
    per-key decay on the token-sequential kernel."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    inp = workloads.workload(name)
    _check(inp, inp.spec.rule, name)
