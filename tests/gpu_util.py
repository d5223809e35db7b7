"""Helpers for the GPU parity tests: move drawn inputs to the device, call the
library through its binding, and measure the spec error metric."""
import numpy as np
import torch

TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-2}

# Bytes of one chunk record (one 64-token chunk and value head) of the tensor-core
# prefill's workspace, as include/gdn.h states it.
RECORD_BYTES = 66560


def rel_err(gpu, ref) -> float:
    """max |gpu - ref| / max |ref| (the parity metric)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    denom = np.max(np.abs(ref))
    diff = np.max(np.abs(gpu - ref))
    if not np.isfinite(diff):
        return float("inf")
    return float(diff / denom) if denom > 0 else float(diff)


def to_device(inp, device="cuda"):
    d = {n: getattr(inp, n).to(device) for n in ("q", "k", "v", "a", "b", "A_log", "dt_bias")}
    d["state_in"] = None if inp.state_in is None else inp.state_in.to(device)
    d["cu_seqlens"] = None
    if inp.varlen:
        d["cu_seqlens"] = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=device)
    return d


def run_prefill(inp, device="cuda", **kw):
    from recurrent_state_scan_gb300 import gdn_prefill
    d = to_device(inp, device)
    o, s = gdn_prefill(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"], d["dt_bias"],
                       d["state_in"], d["cu_seqlens"], inp.scale, **kw)
    torch.cuda.synchronize()
    from recurrent_state_scan_gb300 import gdn_last_device_status
    assert gdn_last_device_status() == 0, "the device check word is set (a bounded wait gave up)"
    spec = inp.spec
    o = o.float().cpu().numpy().reshape(-1, spec.h_v, spec.d_v)
    s = s.cpu().numpy()
    return o, s


def check(inp, o_gpu, s_gpu, o_ref, s_ref, units=None, what=""):
    """Assert parity for all units, or only for the listed (n * h_v + h) ones."""
    tol = TOL[inp.spec.io]
    cu = inp.cu_seqlens
    h_v = inp.spec.h_v
    if units is not None:
        o_sel, o_r, s_sel, s_r = [], [], [], []
        for u in units:
            n, h = divmod(u, h_v)
            o_sel.append(o_gpu[cu[n]:cu[n + 1], h])
            o_r.append(o_ref[cu[n]:cu[n + 1], h])
            s_sel.append(s_gpu[n, h])
            s_r.append(s_ref[n, h])
        o_gpu, o_ref = np.concatenate(o_sel), np.concatenate(o_r)
        s_gpu, s_ref = np.stack(s_sel), np.stack(s_r)
    eo, es = rel_err(o_gpu, o_ref), rel_err(s_gpu, s_ref)
    assert eo <= tol, f"{what} output rel err {eo:.3e} > {tol}"
    assert es <= tol, f"{what} state rel err {es:.3e} > {tol}"
    return eo, es
