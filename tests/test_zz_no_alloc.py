"""gdn_prefill_noalloc, the prefill entry point for callers that may not allocate
device memory (a plugin whose host engine owns the whole memory budget, or a
latency-bound caller that cannot take cudaMalloc's device synchronisation).

Its scratch is a fixed array inside the library, shared by every call on a device
and holding whatever the previous call left there.  The GPU test makes two calls
in a row on the same shape with different inputs, so the second call starts from
the first call's records, and checks each against gdn_prefill (caller-provided
workspace) and against the float64 CPU oracle on the same inputs, within the parity
tolerance of the I/O type.  The file is named to be collected last, and passes alone
or after the other tests.
"""
import ctypes
import os

import pytest
import torch

import oracle
import workloads
from gpu_util import RECORD_BYTES, TOL, check, rel_err, to_device


def test_noalloc_rejects_oversized_shapes_on_the_host():
    from recurrent_state_scan_gb300 import gdn
    lib = gdn.load()
    # 1 x 8192 tokens x 16 value heads needs 128 chunks x 16 records: above 96 MiB.
    shape = gdn.make_shape(gdn.GDN_BF16, 1, 8192, 1, 16, 16, 128, 128)
    assert gdn.gdn_prefill_workspace_bytes(shape) > gdn.PREFILL_NOALLOC_SCRATCH_BYTES
    st = lib.gdn_prefill_noalloc(ctypes.byref(shape), *([None] * 9), 0.0, None, None, None)
    assert st == gdn.GDN_ERR_INVALID_ARG
    assert b"above the fixed" in lib.gdn_last_error_message()
    # The largest advertised example passes the size check: one 4096-token sequence at 16
    # value heads needs 64 x 16 records (the call then stops at its NULL inputs, or at the
    # missing device).  gdn_prefill's own workspace query also counts the time-parallel
    # buffers, which this entry point never uses.
    fits = gdn.make_shape(gdn.GDN_BF16, 1, 4096, 1, 16, 16, 128, 128)
    assert 64 * 16 * RECORD_BYTES <= gdn.PREFILL_NOALLOC_SCRATCH_BYTES
    st = lib.gdn_prefill_noalloc(ctypes.byref(fits), *([None] * 9), 0.0, None, None, None)
    assert st != gdn.GDN_OK and b"above the fixed" not in lib.gdn_last_error_message()


def test_record_size_is_the_documented_one():
    """Two sequences of one chunk at one value head, batched: the workspace is exactly two
    records.  (A batch of one is sized the packed way, two spare records per head.)"""
    from recurrent_state_scan_gb300 import gdn
    two = gdn.make_shape(gdn.GDN_BF16, 2, 64, 2, 1, 1, 128, 128)
    assert gdn.gdn_prefill_workspace_bytes(two) == 2 * RECORD_BYTES
    one = gdn.make_shape(gdn.GDN_BF16, 1, 64, 1, 1, 1, 128, 128)
    assert gdn.gdn_prefill_workspace_bytes(one) == 3 * RECORD_BYTES


def test_noalloc_size_boundary_follows_the_call_layout():
    """A batched call (no cu_seqlens) is sized as batch * ceil(T / 64) * h_v records of
    66,560 bytes: 6,016 tokens at 16 value heads (1,504 records) fit the 96 MiB array
    (1,512 records) and 6,017 (1,520 records) do not.  A packed call of the same tokens
    needs (floor(T / 64) + N + 1) * h_v records."""
    from recurrent_state_scan_gb300 import gdn
    lib = gdn.load()
    rec = RECORD_BYTES
    assert 1512 * rec <= gdn.PREFILL_NOALLOC_SCRATCH_BYTES < 1513 * rec
    for T, fits in ((6016, True), (6017, False)):
        shape = gdn.make_shape(gdn.GDN_BF16, 1, T, 1, 16, 16, 128, 128)
        st = lib.gdn_prefill_noalloc(ctypes.byref(shape), *([None] * 9), 0.0, None, None, None)
        assert st != gdn.GDN_OK
        assert (b"above the fixed" in lib.gdn_last_error_message()) == (not fits), T
    # Packed, one sequence of 5,951 tokens: (92 + 1 + 1) * 16 = 1,504 records fit; a
    # packed 5,952 would need (93 + 2) * 16 = 1,520 and is refused before any pointer is read.
    cu = ctypes.c_void_p(16)   # never dereferenced: the size check comes first
    for T, fits in ((5951, True), (5952, False)):
        shape = gdn.make_shape(gdn.GDN_BF16, 1, T, 1, 16, 16, 128, 128)
        args = [None] * 9
        args[8] = cu
        st = lib.gdn_prefill_noalloc(ctypes.byref(shape), *args, 0.0, None, None, None)
        assert st != gdn.GDN_OK
        assert (b"above the fixed" in lib.gdn_last_error_message()) == (not fits), T


@pytest.mark.gpu
def test_noalloc_matches_gdn_prefill_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import (gdn_last_device_status, gdn_prefill,
                                            gdn_prefill_noalloc, load)
    load()
    tol = TOL["bf16"]
    for seed in (11, 12):
        # Three packed sequences (5, 1 and 3 chunks, two with ragged tails), GQA 2 -> 4.
        inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[300, 64, 129], h_qk=2,
                                                  h_v=4, seed=seed, state_std=0.05))
        d = to_device(inp)
        args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["state_in"],
                d["cu_seqlens"], inp.scale)
        o_ref, s_ref = gdn_prefill(*args)
        o = torch.empty_like(o_ref)
        s = torch.empty_like(s_ref)
        gdn_prefill_noalloc(*args, o=o, state_out=s)
        torch.cuda.synchronize()
        assert gdn_last_device_status() == 0
        eo = rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy())
        es = rel_err(s.cpu().numpy(), s_ref.cpu().numpy())
        assert eo <= tol and es <= tol, f"call with seed {seed}: rel err o {eo:.2e}, state {es:.2e}"
        o_or, s_or = oracle.scan_inputs(inp, threads=4)
        check(inp, o.float().cpu().numpy().reshape(-1, inp.spec.h_v, inp.spec.d_v),
              s.cpu().numpy(), o_or, s_or, what=f"noalloc call with seed {seed} vs oracle")


@pytest.mark.gpu
def test_noalloc_runs_the_largest_advertised_shape():
    """One 4096-token sequence at 16 value heads (the bf16 prefill workload) fits the fixed
    scratch and matches gdn_prefill, which runs the time-parallel scan on that shape."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from recurrent_state_scan_gb300 import (gdn_last_device_status, gdn_prefill,
                                            gdn_prefill_noalloc, load)
    load()
    inp = workloads.workload("bf16_prefill_t4096")
    d = to_device(inp)
    args = (d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"], d["state_in"],
            d["cu_seqlens"], inp.scale)
    o_ref, s_ref = gdn_prefill(*args)
    o = torch.empty_like(o_ref)
    s = torch.empty_like(s_ref)
    gdn_prefill_noalloc(*args, o=o, state_out=s)
    torch.cuda.synchronize()
    assert gdn_last_device_status() == 0
    tol = TOL["bf16"]
    assert rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= tol
    assert rel_err(s.cpu().numpy(), s_ref.cpu().numpy()) <= tol
    o_or, s_or = oracle.scan_inputs(inp, threads=os.cpu_count() or 1)
    check(inp, o.float().cpu().numpy().reshape(-1, inp.spec.h_v, inp.spec.d_v), s.cpu().numpy(),
          o_or, s_or, what="noalloc bf16 prefill T=4096 vs oracle")
