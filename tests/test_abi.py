"""Host-side checks of libgdn's C ABI: no GPU needed, no kernel launched.

The library must load, export every function include/gdn.h declares, and turn
bad arguments into status codes before touching the device.
"""
import ctypes
import os
import re

import pytest

from recurrent_state_scan_gb300 import gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    lib = gdn.load()
    declared = _declared_functions()
    assert "gdn_prefill" in declared and "gdn_decode_step" in declared
    for name in declared:
        assert hasattr(lib, name), f"libgdn does not export {name}"
    assert set(declared) == set(gdn.EXPORTS)


def test_status_strings():
    assert gdn.gdn_status_string(0) == "GDN_OK"
    assert gdn.gdn_status_string(1) == "GDN_ERR_INVALID_ARG"
    assert gdn.gdn_status_string(2) == "GDN_ERR_UNSUPPORTED"
    assert gdn.gdn_status_string(4) == "GDN_ERR_DEVICE_CHECK"


def _call_prefill(shape, ptr=0x1000, cu=None, state_out=0x2000, scale=0.0):
    lib = gdn.load()
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.gdn_prefill(ctypes.byref(shape), p, p, p, p, p, p, p, None,
                           None if cu is None else ctypes.c_void_p(cu), scale, p,
                           ctypes.c_void_p(state_out) if state_out else None, None, 0, None)


def _shape(**kw):
    base = dict(io_dtype=gdn.GDN_BF16, batch=2, seqlen=8, num_seqs=2, h_qk=2, h_v=4, d_k=128,
                d_v=128)
    base.update(kw)
    return gdn.make_shape(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(io_dtype=7), gdn.GDN_ERR_INVALID_ARG),
    (dict(seqlen=-1), gdn.GDN_ERR_INVALID_ARG),
    (dict(num_seqs=3), gdn.GDN_ERR_INVALID_ARG),          # num_seqs != batch
    (dict(h_v=3), gdn.GDN_ERR_INVALID_ARG),               # h_v % h_qk != 0
    (dict(h_qk=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(d_k=0), gdn.GDN_ERR_INVALID_ARG),
    (dict(d_k=257), gdn.GDN_ERR_UNSUPPORTED),             # above the built maximum
    (dict(d_v=130), gdn.GDN_ERR_UNSUPPORTED),             # d_v must be a multiple of 4
])
def test_prefill_rejects_bad_shapes_before_launch(kw, status):
    assert _call_prefill(_shape(**kw)) == status
    assert gdn.load().gdn_last_error_message().decode() != ""


def test_prefill_rejects_null_and_misaligned_pointers():
    assert _call_prefill(_shape(), ptr=0) == gdn.GDN_ERR_INVALID_ARG            # q NULL
    assert _call_prefill(_shape(), ptr=0x1001) == gdn.GDN_ERR_INVALID_ARG       # odd bf16 address
    assert _call_prefill(_shape(), state_out=0) == gdn.GDN_ERR_INVALID_ARG
    assert _call_prefill(_shape(), state_out=0x2004) == gdn.GDN_ERR_INVALID_ARG  # not 16 B
    assert _call_prefill(_shape(), scale=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    # varlen needs batch == 1
    assert _call_prefill(_shape(batch=2, num_seqs=2), cu=0x3000) == gdn.GDN_ERR_INVALID_ARG


def test_empty_problem_is_a_no_op():
    # No sequences: nothing to do, and no device call is needed.
    assert _call_prefill(_shape(batch=0, num_seqs=0, seqlen=5), ptr=0, state_out=0) == gdn.GDN_OK


def test_decode_rejects_bad_arguments():
    lib = gdn.load()
    p = ctypes.c_void_p(0x1000)

    def call(shape, state=0x2000):
        return lib.gdn_decode_step(ctypes.byref(shape), p, p, p, p, p, p, p,
                                   ctypes.c_void_p(state) if state else None, 0.0, p, None)

    assert call(_shape(seqlen=2)) == gdn.GDN_ERR_INVALID_ARG
    assert call(_shape(seqlen=1), state=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(_shape(seqlen=1, h_v=5, h_qk=2)) == gdn.GDN_ERR_INVALID_ARG
    assert call(_shape(seqlen=1, d_k=300)) == gdn.GDN_ERR_UNSUPPORTED


def test_workspace_query_is_host_only():
    assert gdn.gdn_prefill_workspace_bytes(_shape()) >= 0


def test_variant_rejects_bad_rules_and_missing_gates():
    lib = gdn.load()
    p = ctypes.c_void_p(0x1000)

    def call(rule, a=p, b=p, A=p, decay_per_key=0, beta_shared=0, variant=True):
        var = gdn.GdnVariant(rule, decay_per_key, beta_shared)
        return lib.gdn_scan_variant(ctypes.byref(_shape()), ctypes.byref(var) if variant else None,
                                    p, p, p, a, b, A, A, None, None, 0.0, p,
                                    ctypes.c_void_p(0x2000), None)

    assert call(4) == gdn.GDN_ERR_INVALID_ARG                       # no such rule
    assert call(-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(0, variant=False) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.RULES["gated_delta"], b=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.RULES["gated_delta"], a=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.RULES["gated"], A=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.RULES["delta"], b=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.RULES["linear"], a=ctypes.c_void_p(0x1001)) == gdn.GDN_ERR_INVALID_ARG
