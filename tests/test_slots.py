"""GPU parity of gdn_decode_step_slots, the decode step against a pool of states
(nuvec-core src/fast/imp.rs, gated_delta_slots), with the CPU oracle's slot_scan.

Tolerance as in test_parity: max|gpu - ref| / max|ref| <= 1e-4 (fp32 I/O) or 2e-2
(bf16/f16 I/O), on o and on the pool.  Pool entries no slot names must come back
bit-identical.
"""
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


def _run(inp, slots=None):
    from recurrent_state_scan_gb300 import gdn_decode_step_slots, gdn_last_device_status
    d = {n: getattr(inp, n).cuda() for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    pool = inp.pool.cuda().clone()
    sl = (inp.slots if slots is None else torch.as_tensor(slots, dtype=torch.int32)).cuda()
    o = torch.full(d["v"].shape, 7.0, dtype=d["v"].dtype, device="cuda")   # sentinel
    gdn_decode_step_slots(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                          pool, sl, inp.scale, o=o)
    status = gdn_last_device_status()
    s = inp.spec
    return o.float().cpu().numpy().reshape(-1, s.h_v, s.d_v), pool.cpu().numpy(), status


def _ref(inp, slots):
    s, f = inp.spec, inp.f64
    return oracle.slot_scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"],
                            f["a"], f["b"], f["A_log"], f["dt_bias"], f["pool"], slots,
                            scale=inp.scale, threads=4)


@pytest.mark.parametrize("io", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("dims", [(6, 2, 4, 128, 128), (5, 1, 2, 64, 32), (3, 2, 2, 256, 256)])
def test_slot_decode_matches_oracle(io, dims):
    n, h_qk, h_v, d_k, d_v = dims
    inp = workloads.draw(workloads.small_spec(io=io, batch=n, seqlen=1, h_qk=h_qk, h_v=h_v,
                                              d_k=d_k, d_v=d_v, decode=True, pool_size=2 * n + 1,
                                              pool_std=0.05, seed=71 + n))
    slots = inp.slots.numpy()
    o, pool, status = _run(inp)
    o_ref, pool_ref = _ref(inp, slots)
    assert status == 0
    tol = TOL[io]
    assert rel_err(o, o_ref) <= tol
    assert rel_err(pool[slots], pool_ref[slots]) <= tol
    untouched = sorted(set(range(2 * n + 1)) - set(int(x) for x in slots))
    assert np.array_equal(pool[untouched], inp.pool.numpy()[untouched])


def test_slot_outside_the_pool_skips_its_row_and_sets_the_check_word():
    from recurrent_state_scan_gb300 import gdn
    inp = workloads.draw(workloads.small_spec(io="bf16", batch=4, seqlen=1, h_qk=2, h_v=2,
                                              decode=True, pool_size=6, pool_std=0.05, seed=81))
    slots = inp.slots.numpy().copy()
    slots[1] = -1
    o, pool, status = _run(inp, slots)
    assert status == gdn.GDN_ERR_DEVICE_CHECK
    o_ref, pool_ref = _ref(inp, slots)
    keep = [0, 2, 3]
    assert rel_err(o[keep], o_ref[keep]) <= TOL["bf16"]
    assert np.all(o[1] == 7.0)                     # the skipped row is left as it was
    named = [int(slots[i]) for i in keep]
    assert rel_err(pool[named], pool_ref[named]) <= TOL["bf16"]
    others = sorted(set(range(6)) - set(named))
    assert np.array_equal(pool[others], inp.pool.numpy()[others])


def test_slot_decode_full_size_workload():
    inp = workloads.workload("bf16_slot_decode_b256")
    slots = inp.slots.numpy()
    o, pool, status = _run(inp)
    o_ref, pool_ref = _ref(inp, slots)
    assert status == 0
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(pool[slots], pool_ref[slots]) <= TOL["bf16"]
    untouched = sorted(set(range(inp.spec.pool_size)) - set(int(x) for x in slots))
    assert np.array_equal(pool[untouched], inp.pool.numpy()[untouched])
