"""GPU parity of gdn_scan_variant -- the update rules (gated_delta, delta, gated,
linear), one decay per key dimension and one beta shared by every head -- with the CPU
oracle run on the same drawn inputs.  Tolerances as in test_parity."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

RULES = ("gated_delta", "delta", "gated", "linear")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _run(inp, rule, in_place=False):
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_scan_variant
    s = inp.spec
    d = to_device(inp)
    st = d["state_in"]
    o, state = gdn_scan_variant(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], st, d["cu_seqlens"], inp.scale, rule=rule,
                                decay_per_key=s.decay_per_key, beta_shared=s.beta_shared,
                                state_out=st if in_place else None)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    return o.float().cpu().numpy().reshape(-1, s.h_v, s.d_v), state.cpu().numpy()


def _check(inp, rule, **kw):
    o, s = _run(inp, rule, **kw)
    o_ref, s_ref = oracle.scan_inputs(inp, rule=rule, threads=4)
    tol = TOL[inp.spec.io]
    assert rel_err(o, o_ref) <= tol, "o"
    assert rel_err(s, s_ref) <= tol, "state"


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("rule", RULES)
def test_rules_match_oracle(io, rule):
    inp = workloads.draw(workloads.small_spec(io=io, batch=2, seqlen=37, h_qk=2, h_v=4,
                                              state_std=0.05, seed=301))
    _check(inp, rule)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("rule", ["gated_delta", "gated"])
def test_per_key_decay_varlen(io, rule):
    inp = workloads.draw(workloads.small_spec(io=io, lengths=(1, 29, 64, 7), h_qk=2, h_v=4,
                                              state_std=0.05, seed=302, decay_per_key=True))
    _check(inp, rule)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("rule", ["gated_delta", "delta"])
def test_shared_beta(io, rule):
    inp = workloads.draw(workloads.small_spec(io=io, batch=3, seqlen=20, h_qk=1, h_v=4,
                                              state_std=0.05, seed=303, beta_shared=True))
    _check(inp, rule)


def test_per_key_decay_and_shared_beta_with_small_heads():
    inp = workloads.draw(workloads.small_spec(io="f32", batch=2, seqlen=33, h_qk=2, h_v=2,
                                              d_k=64, d_v=96, state_std=0.05, seed=304,
                                              decay_per_key=True, beta_shared=True))
    _check(inp, "gated_delta")


@pytest.mark.parametrize("rule", RULES)
def test_decode_step_in_place(rule):
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=5, seqlen=1, h_qk=2, h_v=4,
                                              state_std=0.05, seed=305, decode=True,
                                              decay_per_key=True))
    _check(inp, rule, in_place=True)


def test_empty_sequences_keep_their_state():
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=(0, 5, 0), h_qk=2, h_v=2,
                                              state_std=0.05, seed=306, decay_per_key=True))
    o, s = _run(inp, "gated_delta")
    assert np.array_equal(s[0], inp.state_in[0].numpy())
    assert np.array_equal(s[2], inp.state_in[2].numpy())
    _check(inp, "gated_delta")


def test_per_key_decode_full_size_workload():
    inp = workloads.workload("bf16_perkey_decode_b256")
    o, s = _run(inp, "gated_delta", in_place=True)
    o_ref, s_ref = oracle.scan_inputs(inp, threads=16)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(s, s_ref) <= TOL["bf16"]
