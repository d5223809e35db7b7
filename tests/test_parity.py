"""GPU parity: libgdn (through its C ABI) against the float64 CPU oracle.

Tolerance (max|gpu - ref| / max|ref|, separately for o and the final state):
1e-4 for fp32 I/O, 2e-2 for bf16/f16 I/O; the state is fp32 on both sides.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import RECORD_BYTES, TOL, check, rel_err, run_prefill, to_device

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import load
    load()


def _decode(inp, state=None):
    from recurrent_state_scan_gb300 import gdn_decode_step
    d = to_device(inp)
    st = d["state_in"].clone() if state is None else state
    o = gdn_decode_step(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], st,
                        inp.scale)
    torch.cuda.synchronize()
    return o.float().cpu().numpy().reshape(-1, inp.spec.h_v, inp.spec.d_v), st.cpu().numpy()


# ---------------------------------------------------------------- measured workloads

def test_tiny_f32_prefill_full():
    inp = workloads.workload("tiny_f32_prefill")
    o_ref, s_ref = oracle.scan_inputs(inp)
    o, s = run_prefill(inp)
    check(inp, o, s, o_ref, s_ref, what="tiny fp32 prefill")


def test_decode_b256_full():
    inp = workloads.workload("bf16_decode_b256")
    o_ref, s_ref = oracle.scan_inputs(inp, threads=8)
    o, s = _decode(inp)
    check(inp, o, s, o_ref, s_ref, what="decode B=256")


FULL_SIZE_PREFILL = ["bf16_prefill_t4096", "varlen_bf16_prefill", "gqa_f16_prefill"]


@pytest.mark.parametrize("name", FULL_SIZE_PREFILL)
def test_prefill_workloads_full(name):
    """Full-size run in the benchmark's launch configuration against the oracle over the
    whole workload: every token of every (sequence, head) unit and every final state."""
    import os
    inp = workloads.workload(name)
    o, s = run_prefill(inp)
    o_ref, s_ref = oracle.scan_inputs(inp, threads=os.cpu_count() or 1)
    eo, es = check(inp, o, s, o_ref, s_ref, what=name)
    print(f"{name}: max|d|/max|ref| o {eo:.3e}, state {es:.3e}")


# ---------------------------------------------------------------- small shapes, edges

@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("dims", [(2, 4, 128, 128), (1, 1, 64, 32), (2, 2, 256, 256),
                                  (3, 3, 100, 36), (1, 2, 32, 4)])
def test_decode_small(io, dims):
    h_qk, h_v, d_k, d_v = dims
    inp = workloads.draw(workloads.small_spec(io=io, batch=5, seqlen=1, h_qk=h_qk, h_v=h_v,
                                              d_k=d_k, d_v=d_v, seed=31, state_std=0.05,
                                              decode=True))
    o_ref, s_ref = oracle.scan_inputs(inp)
    o, s = _decode(inp)
    check(inp, o, s, o_ref, s_ref, what=f"decode {io} {dims}")


PREFILL_CASES = [
    # (io, lengths, h_qk, h_v, d_k, d_v, state_std)
    ("bf16", [64], 1, 1, 128, 128, 0.0),
    ("bf16", [1, 63, 65, 130, 0, 200], 2, 2, 128, 128, 0.05),   # ragged chunks, empty seq
    ("f16", [129, 64, 7], 2, 4, 128, 128, 0.05),                # GQA
    ("bf16", [300], 1, 1, 128, 128, 0.0),
    ("f32", [64, 33], 2, 2, 32, 32, 0.0),
    ("f32", [100], 1, 2, 128, 128, 0.05),
    ("bf16", [50, 20], 1, 1, 64, 64, 0.05),
    ("f16", [40], 2, 2, 256, 128, 0.05),
    ("bf16", [17, 0, 0, 5], 1, 1, 96, 12, 0.05),
    ("bf16", [70, 1, 130, 64], 16, 32, 128, 128, 0.05),        # >= 120 units: 128-column CTAs
    ("f16", [200, 3], 8, 64, 128, 128, 0.0),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: f"{c[0]}-{len(c[1])}seq-d{c[4]}x{c[5]}")
def test_prefill_small(case):
    io, lengths, h_qk, h_v, d_k, d_v, sstd = case
    inp = workloads.draw(workloads.small_spec(io=io, lengths=lengths, h_qk=h_qk, h_v=h_v,
                                              d_k=d_k, d_v=d_v, seed=41 + len(lengths),
                                              state_std=sstd))
    o_ref, s_ref = oracle.scan_inputs(inp)
    o, s = run_prefill(inp)
    check(inp, o, s, o_ref, s_ref, what=f"prefill {case}")


def test_plan_takes_the_tensor_core_path_for_16bit_d128():
    from recurrent_state_scan_gb300 import gdn
    for io in (gdn.GDN_BF16, gdn.GDN_F16):
        assert gdn.gdn_prefill_plan(gdn.make_shape(io, 1, 4096, 1, 16, 16, 128, 128))[0] in \
            (gdn.PATH_TC, gdn.PATH_TC_TP)
    assert gdn.gdn_prefill_plan(gdn.make_shape(gdn.GDN_F32, 1, 64, 1, 2, 2, 32, 32))[0] == gdn.PATH_SIMT
    assert gdn.gdn_prefill_plan(gdn.make_shape(gdn.GDN_BF16, 1, 64, 1, 2, 2, 64, 64))[0] == gdn.PATH_SIMT


def test_prefill_batched_equals_varlen():
    """B sequences of one length through the batched layout and through cu_seqlens."""
    spec = workloads.small_spec(io="bf16", batch=3, seqlen=150, h_qk=2, h_v=2, seed=51,
                                state_std=0.05)
    inp = workloads.draw(spec)
    o_ref, s_ref = oracle.scan_inputs(inp)
    o, s = run_prefill(inp)
    check(inp, o, s, o_ref, s_ref, what="batched")
    from recurrent_state_scan_gb300 import gdn_prefill
    d = to_device(inp)
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
    flat = {n: d[n].reshape(1, -1, *d[n].shape[2:]) for n in ("q", "k", "v", "a", "b")}
    o2, s2 = gdn_prefill(flat["q"], flat["k"], flat["v"], flat["a"], flat["b"], d["A_log"],
                         d["dt_bias"], d["state_in"], cu, inp.scale)
    o2 = o2.float().cpu().numpy().reshape(o.shape)
    assert rel_err(o2, o_ref) <= TOL["bf16"] and rel_err(s2.cpu().numpy(), s_ref) <= TOL["bf16"]


def test_chaining_and_decode_steps():
    """prefill(T1) then prefill(T2) from its state, and T decode steps, all equal
    one prefill over T1+T2 (each within tolerance of the oracle)."""
    from recurrent_state_scan_gb300 import gdn_decode_step, gdn_prefill
    spec = workloads.small_spec(io="bf16", batch=2, seqlen=96, h_qk=1, h_v=2, seed=61,
                                state_std=0.05)
    inp = workloads.draw(spec)
    o_ref, s_ref = oracle.scan_inputs(inp)
    d = to_device(inp)
    T1 = 40
    sl = lambda x, a, b: x[:, a:b].contiguous()
    oa, sa = gdn_prefill(*(sl(d[n], 0, T1) for n in ("q", "k", "v", "a", "b")), d["A_log"],
                         d["dt_bias"], d["state_in"], None, inp.scale)
    ob, sb = gdn_prefill(*(sl(d[n], T1, 96) for n in ("q", "k", "v", "a", "b")), d["A_log"],
                         d["dt_bias"], sa, None, inp.scale)
    o = torch.cat([oa, ob], dim=1).float().cpu().numpy().reshape(-1, 2, 128)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(sb.cpu().numpy(), s_ref) <= TOL["bf16"]
    st = d["state_in"].clone()
    outs = []
    for t in range(96):
        outs.append(gdn_decode_step(*(sl(d[n], t, t + 1) for n in ("q", "k", "v", "a", "b")),
                                    d["A_log"], d["dt_bias"], st, inp.scale))
    o = torch.cat(outs, dim=1).float().cpu().numpy().reshape(-1, 2, 128)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(st.cpu().numpy(), s_ref) <= TOL["bf16"]


def test_state_in_place_and_null_state():
    from recurrent_state_scan_gb300 import gdn_prefill
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[70, 0, 9], seed=71,
                                              state_std=0.05))
    o_ref, s_ref = oracle.scan_inputs(inp)
    d = to_device(inp)
    st = d["state_in"].clone()
    o, s = gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], st,
                       d["cu_seqlens"], inp.scale, state_out=st)
    assert s.data_ptr() == st.data_ptr()
    assert rel_err(st.cpu().numpy(), s_ref) <= TOL["bf16"]
    # The empty sequence keeps its state exactly.
    assert np.array_equal(st.cpu().numpy()[1], inp.state_in.numpy()[1])
    # NULL state_in means zeros.
    o0, s0 = gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], None,
                         d["cu_seqlens"], inp.scale)
    f = inp.f64
    o_ref0, s_ref0 = oracle.scan(inp.cu_seqlens, 2, 2, 128, 128, f["q"], f["k"], f["v"],
                                 a=f["a"], b=f["b"], A_log=f["A_log"], dt_bias=f["dt_bias"],
                                 scale=inp.scale)
    assert rel_err(s0.cpu().numpy(), s_ref0) <= TOL["bf16"]
    assert np.all(s0.cpu().numpy()[1] == 0.0)


def test_zero_gates_invariant_on_gpu():
    """b = -inf (beta = 0) and A_log = -inf (g = 0): o = 0 and S = 0 from a zero state."""
    from recurrent_state_scan_gb300 import gdn_prefill
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[130], seed=81))
    d = to_device(inp)
    d["b"].fill_(float("-inf"))
    A_log = torch.full_like(d["A_log"], float("-inf"))
    o, s = gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], A_log, d["dt_bias"], None,
                       d["cu_seqlens"], inp.scale)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(s == 0)


def test_bad_device_cu_seqlens_sets_check_word():
    """A malformed device cu_seqlens is skipped and reported, without a fault."""
    from recurrent_state_scan_gb300 import gdn_last_device_status, gdn_prefill
    from recurrent_state_scan_gb300.gdn import GDN_ERR_DEVICE_CHECK, GDN_OK
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[10, 20], seed=91))
    d = to_device(inp)
    assert gdn_last_device_status() == GDN_OK
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")   # decreasing
    gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], None, bad,
                inp.scale)
    assert gdn_last_device_status() == GDN_ERR_DEVICE_CHECK
    assert gdn_last_device_status() == GDN_OK          # read-and-clear
    o, s = run_prefill(inp)                            # the context is still usable
    o_ref, s_ref = oracle.scan_inputs(inp)
    check(inp, o, s, o_ref, s_ref, what="after device check")


def test_prefill_time_parallel_with_ragged_tail():
    """A batched call with a small scan grid and 65 chunks runs the time-parallel scan: four
    segments of 17 chunks (the last one 14, its last chunk ragged), each scanned from zero
    beside its operator pass, then combined and corrected; against the oracle, with an
    initial state.  The plan reports prep, scan, three combine steps and the correction."""
    from recurrent_state_scan_gb300 import gdn
    spec = workloads.small_spec(io="bf16", batch=1, seqlen=4100, h_qk=2, h_v=4, seed=61,
                                state_std=0.05)
    inp = workloads.draw(spec)
    path, launches = gdn.gdn_prefill_plan(gdn.shape_of_spec(spec, inp.n_seq, inp.total_tokens))
    assert path == gdn.PATH_TC_TP and launches == 6
    o_ref, s_ref = oracle.scan_inputs(inp, threads=4)
    o, s = run_prefill(inp)
    check(inp, o, s, o_ref, s_ref, what="time-parallel scan")


@pytest.mark.parametrize("io,B,T,hqk,hv,state", [
    ("f16", 2, 2048, 2, 2, False),     # two segments of 16 chunks
    ("bf16", 1, 3000, 1, 2, True),     # GQA, ragged tail
    ("bf16", 3, 4096, 2, 2, True),     # three sequences, four segments
])
def test_prefill_time_parallel_shapes(io, B, T, hqk, hv, state):
    spec = workloads.small_spec(io=io, batch=B, seqlen=T, h_qk=hqk, h_v=hv, seed=62 + T,
                                state_std=0.05 if state else 0.0)
    inp = workloads.draw(spec)
    o_ref, s_ref = oracle.scan_inputs(inp, threads=8)
    o, s = run_prefill(inp)
    check(inp, o, s, o_ref, s_ref, what="time-parallel scan")


def test_prefill_time_segments_with_a_records_only_workspace():
    """Given room for the chunk records only (65 KiB per chunk and value head), the same
    call falls back to the overlapped prep/scan segments, with the same results."""
    spec = workloads.small_spec(io="bf16", batch=1, seqlen=4100, h_qk=2, h_v=4, seed=61,
                                state_std=0.05)
    inp = workloads.draw(spec)
    records = ((4100 + 63) // 64) * 4 * RECORD_BYTES
    ws = torch.empty(records, dtype=torch.uint8, device="cuda")
    o_ref, s_ref = oracle.scan_inputs(inp, threads=4)
    o, s = run_prefill(inp, workspace=ws)
    check(inp, o, s, o_ref, s_ref, what="overlapped segments")


def test_time_parallel_error_next_to_the_sequential_chain():
    """On the 4096-token bf16 prefill the time-parallel path (segments scanned at once, then
    o += R S_k with S_k in fp32) and the sequential chain over the chunk records (a
    records-only workspace) are both compared with the oracle; the time-parallel path may
    not lose more than a third of a bf16 rounding step on top of the chain's error."""
    import os
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.workload("bf16_prefill_t4096")
    shape = gdn.shape_of_spec(inp.spec, inp.n_seq, inp.total_tokens)
    assert gdn.gdn_prefill_plan(shape)[0] == gdn.PATH_TC_TP
    o_ref, s_ref = oracle.scan_inputs(inp, threads=os.cpu_count() or 1)
    o_tp, s_tp = run_prefill(inp)
    records = ((4096 // 64) + 1 + 1) * 16 * RECORD_BYTES
    o_ch, s_ch = run_prefill(inp, workspace=torch.empty(records, dtype=torch.uint8, device="cuda"))
    e_tp = (rel_err(o_tp, o_ref), rel_err(s_tp, s_ref))
    e_ch = (rel_err(o_ch, o_ref), rel_err(s_ch, s_ref))
    print(f"time-parallel: o {e_tp[0]:.3e} state {e_tp[1]:.3e}; sequential chain: o {e_ch[0]:.3e} "
          f"state {e_ch[1]:.3e}")
    assert max(e_tp + e_ch) <= TOL["bf16"]
    assert e_tp[0] <= e_ch[0] + 2 ** -9 / 3 and e_tp[1] <= e_ch[1] + 2 ** -9 / 3
