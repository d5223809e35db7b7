"""The tensor-core prefill's bounded waits, made to run out on purpose.

Every wait in the chunk-prep and state-scan kernels gives up after a cycle budget: the
CTA then lets the copies and MMAs it has issued finish (under the full budget), frees
its tensor memory, sets the device check word and leaves.  gdn_set_wait_budget shortens
the budget of the waits on work in flight (not of those drains), so a small prefill
times out without anything being stalled: its loads and MMAs simply take longer than
the budget.  The call must then report GDN_ERR_TIMEOUT, leave nothing running, and a
normal call afterwards must match the oracle.
"""
import pytest
import torch

import oracle
import workloads
from gpu_util import check, run_prefill, to_device

def test_set_wait_budget_rejects_negative_values():
    from recurrent_state_scan_gb300 import gdn
    with pytest.raises(gdn.GdnError):
        gdn.gdn_set_wait_budget(-1)


@pytest.mark.gpu
def test_short_wait_budget_reports_timeout_then_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn, gdn_last_device_status, gdn_prefill
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[300, 130], h_qk=1, h_v=2,
                                              seed=17, state_std=0.05))
    assert gdn.gdn_prefill_plan(gdn.shape_of_spec(inp.spec, inp.n_seq, inp.total_tokens))[0] == \
        gdn.PATH_TC
    d = to_device(inp)
    assert gdn_last_device_status() == gdn.GDN_OK
    gdn.gdn_set_wait_budget(200)          # far below one MMA group or one tile load
    try:
        gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                    d["state_in"], d["cu_seqlens"], inp.scale)
        torch.cuda.synchronize()          # every CTA has left: nothing is left waiting
        assert gdn_last_device_status() == gdn.GDN_ERR_TIMEOUT
    finally:
        gdn.gdn_set_wait_budget(0)
    assert gdn_last_device_status() == gdn.GDN_OK      # read-and-clear
    o, s = run_prefill(inp)
    o_ref, s_ref = oracle.scan_inputs(inp)
    check(inp, o, s, o_ref, s_ref, what="prefill after a timed-out call")
