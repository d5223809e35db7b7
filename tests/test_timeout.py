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


@pytest.mark.gpu
def test_short_wait_budget_times_out_the_conv_pipeline_then_recovers():
    """The bulk-copy causal conv (16-bit long rows) waits for each stage's copies with the
    same budget.  Its stages are prefetched three deep, so only a CTA's first wait can run
    long; rows larger than L2 make those first copies come from DRAM, past a 50-cycle
    budget.  The CTAs then give up, let their copies land and report GDN_ERR_TIMEOUT; the
    next call is exact again (checked on the first 300 tokens of row 0, which depend on
    nothing later)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import numpy as np
    from recurrent_state_scan_gb300 import gdn, gdn_causal_conv, gdn_last_device_status
    inp = workloads.draw_conv(workloads.ConvSpec("t", "bf16", 4, 8192, 4096, 23, kernel=4,
                                                 silu=True, bias=True, state_std=1.0))
    x, w, b, st = inp.x.cuda(), inp.w.cuda(), inp.bias.cuda(), inp.state_in.cuda()
    torch.empty(256 << 20, dtype=torch.uint8, device="cuda").zero_()   # evict x from L2
    torch.cuda.synchronize()
    assert gdn_last_device_status() == gdn.GDN_OK
    gdn.gdn_set_wait_budget(50)
    try:
        gdn_causal_conv(x, w, b, st, activation="silu")
        torch.cuda.synchronize()
        assert gdn_last_device_status() == gdn.GDN_ERR_TIMEOUT
    finally:
        gdn.gdn_set_wait_budget(0)
    assert gdn_last_device_status() == gdn.GDN_OK
    y, _ = gdn_causal_conv(x, w, b, st, activation="silu")
    torch.cuda.synchronize()
    assert gdn_last_device_status() == gdn.GDN_OK
    xs = inp.x[:1, :300].double().numpy()
    y_ref, _ = oracle.causal_conv(xs, inp.w.double().numpy(), inp.bias.double().numpy(),
                                  inp.state_in[:1].double().numpy(), silu=True)
    ref = np.asarray(y_ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.max(np.abs(ref))
    assert np.all(np.abs(y[:1, :300].double().cpu().numpy() - ref) <= bound)


@pytest.mark.gpu
def test_short_wait_budget_times_out_the_norm_pairs_then_recovers():
    """gdn_prefill_norm fused on the tensor-core path: the scan CTAs run as cluster pairs
    that wait on each other for every chunk's row sums.  Under a short budget the waits run
    out, every CTA of a pair leaves (they meet at the cluster barrier on the way out) and
    the call reports GDN_ERR_TIMEOUT; the next call equals the separate calls."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import (gdn, gdn_gated_rmsnorm, gdn_last_device_status,
                                            gdn_prefill, gdn_prefill_norm)
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[300, 130], h_qk=1, h_v=2,
                                              seed=19, state_std=0.05))
    n = workloads.draw_norm(workloads.NormSpec("t", "bf16", (inp.total_tokens, 2, 128), 20))
    d = to_device(inp)
    scale, gate = n.scale.cuda(), n.gate.cuda().view(d["v"].shape)
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["state_in"],
            d["cu_seqlens"], inp.scale)
    assert gdn_last_device_status() == gdn.GDN_OK
    gdn.gdn_set_wait_budget(200)
    try:
        gdn_prefill_norm(*args, norm_scale=scale, gate=gate, eps=1e-6, fuse=True)
        torch.cuda.synchronize()
        assert gdn_last_device_status() == gdn.GDN_ERR_TIMEOUT
    finally:
        gdn.gdn_set_wait_budget(0)
    assert gdn_last_device_status() == gdn.GDN_OK
    y, st = gdn_prefill_norm(*args, norm_scale=scale, gate=gate, eps=1e-6, fuse=True)
    o, st2 = gdn_prefill(*args)
    y2 = gdn_gated_rmsnorm(o, scale, gate, 1e-6, "silu")
    torch.cuda.synchronize()
    assert gdn_last_device_status() == gdn.GDN_OK
    assert torch.equal(st, st2)
    assert torch.allclose(y.float(), y2.float(), rtol=2.0 ** -7, atol=1e-5)


@pytest.mark.gpu
def test_short_wait_budget_times_out_the_per_key_prep_then_recovers():
    """The per-key-dim decay prefill (its own prep kernel, the scan's per-key form) under
    the same 200-cycle budget, then a normal call against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn, gdn_last_device_status, gdn_prefill_variant
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[300, 130], h_qk=1, h_v=2,
                                              seed=19, state_std=0.05, decay_per_key=True))
    d = to_device(inp)
    assert gdn_last_device_status() == gdn.GDN_OK

    def call():
        return gdn_prefill_variant(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                                   d["state_in"], d["cu_seqlens"], inp.scale, decay_per_key=True)
    gdn.gdn_set_wait_budget(200)
    try:
        call()
        torch.cuda.synchronize()
        assert gdn_last_device_status() == gdn.GDN_ERR_TIMEOUT
    finally:
        gdn.gdn_set_wait_budget(0)
    assert gdn_last_device_status() == gdn.GDN_OK
    o, s = call()
    torch.cuda.synchronize()
    assert gdn_last_device_status() == gdn.GDN_OK
    o_ref, s_ref = oracle.scan_inputs(inp)
    check(inp, o.float().cpu().numpy().reshape(-1, 2, 128), s.cpu().numpy(), o_ref, s_ref,
          what="per-key prefill after a timed-out call")


@pytest.mark.gpu
def test_short_wait_budget_times_out_the_layer_conv_pass_then_recovers():
    """gdn_prefill_layer in its default form: the conv pass waits for each TMA stage of x
    under the same budget (a 17.5 KB copy takes longer than 200 cycles even from L2), then
    the prep and the scan do.  The CTAs give up, let the copies they issued land and
    report GDN_ERR_TIMEOUT; the next call repeats the one made before the timeout bit for
    bit, outputs and both states."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import gdn, gdn_last_device_status, gdn_prefill_layer
    s = workloads.PrefillLayerSpec(name="t", io="bf16", h_qk=2, h_v=4, seed=711,
                                   lengths=(300, 0, 130, 1))
    inp = workloads.draw_prefill_layer(s)
    d = lambda t: None if t is None else t.cuda()
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")

    def call():
        out = gdn_prefill_layer(d(inp.x), d(inp.w), d(inp.bias), d(inp.conv_state), d(inp.a),
                                d(inp.b), d(inp.A_log), d(inp.dt_bias), d(inp.state_in), cu,
                                d(inp.norm_scale), d(inp.gate), h_qk=s.h_qk, h_v=s.h_v,
                                scale=inp.scale, conv_activation="silu" if s.silu else "none",
                                norm_activation=s.activation, eps=s.eps)
        torch.cuda.synchronize()
        return out

    before = call()
    assert gdn_last_device_status() == gdn.GDN_OK
    gdn.gdn_set_wait_budget(200)
    try:
        call()
        assert gdn_last_device_status() == gdn.GDN_ERR_TIMEOUT
    finally:
        gdn.gdn_set_wait_budget(0)
    assert gdn_last_device_status() == gdn.GDN_OK
    after = call()
    assert gdn_last_device_status() == gdn.GDN_OK
    for b, a in zip(before, after):
        assert torch.equal(b, a)
