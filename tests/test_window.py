"""GPU parity of gdn_scan_window (the states after the last W steps, for speculative
decoding) with the CPU oracle's window_scan.  Tolerance as in test_parity, on o and on
every slab of the window; slabs before the first step must be exactly zero."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import TOL, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _run(inp, W):
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_scan_window
    d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    st = None if inp.state_in is None else inp.state_in.cuda()
    window = torch.full((W, inp.spec.batch, inp.spec.h_v, inp.spec.d_k, inp.spec.d_v), 3.0,
                        device="cuda")
    o, window = gdn_scan_window(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], st, inp.scale, window_len=W, window=window)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    s = inp.spec
    return o.float().cpu().numpy().reshape(-1, s.h_v, s.d_v), window.cpu().numpy()


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("btw", [(3, 5, 8), (2, 8, 8), (2, 12, 4), (2, 1, 1)])
def test_window_matches_oracle(io, btw):
    B, T, W = btw
    inp = workloads.draw(workloads.small_spec(io=io, batch=B, seqlen=T, h_qk=2, h_v=4,
                                              state_std=0.05, seed=91 + T, window=W))
    o, win = _run(inp, W)
    s, f = inp.spec, inp.f64
    o_ref, win_ref = oracle.window_scan(B, T, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"],
                                        f["a"], f["b"], f["A_log"], f["dt_bias"], f["state_in"],
                                        W, scale=inp.scale, threads=4)
    tol = TOL[io]
    assert rel_err(o, o_ref) <= tol
    lead = max(W - T, 0)
    assert np.all(win[:lead] == 0.0)
    for w in range(lead, W):
        assert rel_err(win[w], win_ref[w]) <= tol, f"slab {w}"


def test_window_full_size_workload():
    inp = workloads.workload("bf16_window_b256_t4")
    o, win = _run(inp, inp.spec.window)
    o_ref, win_ref = oracle.window_scan_inputs(inp, threads=16)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    for w in range(inp.spec.window):
        assert rel_err(win[w], win_ref[w]) <= TOL["bf16"], f"slab {w}"
