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


def _conv_shape(**kw):
    base = dict(io_dtype=gdn.GDN_BF16, batch=2, seqlen=8, channels=16, kernel=4, dilation=1,
                channels_last=1, activation=1, state_window=0)
    base.update(kw)
    return gdn.GdnConvShape(*[base[n] for n, _ in gdn.GdnConvShape._fields_])


@pytest.mark.parametrize("kw", [
    dict(io_dtype=9), dict(batch=-1), dict(seqlen=-1), dict(channels=0), dict(kernel=0),
    dict(kernel=65), dict(dilation=0), dict(kernel=4, dilation=2000), dict(channels_last=2),
    dict(activation=2), dict(state_window=9), dict(state_window=-1),
])
def test_conv_rejects_bad_geometry_before_launch(kw):
    lib = gdn.load()
    p = ctypes.c_void_p(0x1000)
    assert lib.gdn_causal_conv(ctypes.byref(_conv_shape(**kw)), p, p, p, p, p, p, None) == \
        gdn.GDN_ERR_INVALID_ARG


def test_conv_rejects_null_and_misaligned_pointers():
    lib = gdn.load()
    p, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1001)
    s = ctypes.byref(_conv_shape())
    assert lib.gdn_causal_conv(s, None, p, None, None, p, None, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_causal_conv(s, p, None, None, None, p, None, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_causal_conv(s, p, p, odd, None, p, None, None) == gdn.GDN_ERR_INVALID_ARG
    # The pool form: channels last, no window, slots present.
    assert lib.gdn_causal_conv_slots(ctypes.byref(_conv_shape(channels_last=0)), p, p, None, p, 4,
                                     p, p, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_causal_conv_slots(ctypes.byref(_conv_shape(state_window=2)), p, p, None, p, 4,
                                     p, p, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_causal_conv_slots(s, p, p, None, p, 4, None, p, None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_causal_conv_slots(s, p, p, None, p, -1, p, p, None) == gdn.GDN_ERR_INVALID_ARG
    # No rows: nothing to do.
    assert lib.gdn_causal_conv(ctypes.byref(_conv_shape(batch=0)), None, None, None, None, None,
                               None, None) == gdn.GDN_OK


def test_norm_rejects_bad_arguments_before_launch():
    lib = gdn.load()
    p, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1001)

    def call(io=gdn.GDN_BF16, rows=4, width=128, x=p, eps=1e-6, act=1):
        return lib.gdn_gated_rmsnorm(io, rows, width, x, p, p, eps, act, p, None)

    assert call(io=5) == gdn.GDN_ERR_INVALID_ARG
    assert call(rows=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(width=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(act=0) == gdn.GDN_ERR_INVALID_ARG           # the norm has no "none"
    assert call(eps=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert call(eps=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    assert call(x=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(x=odd) == gdn.GDN_ERR_INVALID_ARG
    assert call(rows=0, x=None) == gdn.GDN_OK


def _header_text():
    text = ""
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text += open(os.path.join(ROOT, "include", fn)).read()
    return re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def test_header_enums_match_the_binding():
    """Every enum value the header defines equals the binding's constant of that name."""
    vals = dict((n, int(v)) for n, v in re.findall(r"\b(GDN_[A-Z0-9_]+)\s*=\s*(\d+)", _header_text()))
    assert {k: vals[k] for k in ("GDN_F32", "GDN_BF16", "GDN_F16")} == \
        {"GDN_F32": gdn.GDN_F32, "GDN_BF16": gdn.GDN_BF16, "GDN_F16": gdn.GDN_F16}
    for name in ("GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED", "GDN_ERR_CUDA",
                 "GDN_ERR_DEVICE_CHECK", "GDN_ERR_TIMEOUT"):
        assert vals[name] == getattr(gdn, name), name
    for rule, code in gdn.RULES.items():
        assert vals["GDN_RULE_" + rule.upper()] == code
    assert vals["GDN_ACT_NONE"] == gdn.ACTIVATIONS["none"]
    assert vals["GDN_ACT_SILU"] == gdn.ACTIVATIONS["silu"]
    assert vals["GDN_ACT_SIGMOID"] == gdn.ACTIVATIONS["sigmoid"]


def test_header_structs_match_the_binding():
    """The ctypes structures list the header's fields in order, with the same widths."""
    text = _header_text()
    for cname, pyclass in (("gdn_shape", gdn.GdnShape), ("gdn_variant", gdn.GdnVariant),
                           ("gdn_conv_shape", gdn.GdnConvShape)):
        body = re.search(r"typedef struct " + cname + r"\s*\{(.*?)\}\s*" + cname + ";", text, re.S)
        assert body, cname
        fields = re.findall(r"(int32_t|int64_t)\s+([a-z_]+)\s*;", body.group(1))
        assert [n for _, n in fields] == [n for n, _ in pyclass._fields_], cname
        widths = {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64}
        assert [widths[t] for t, _ in fields] == [t for _, t in pyclass._fields_], cname


def test_noalloc_scratch_size_matches_the_header():
    m = re.search(r"#define GDN_PREFILL_NOALLOC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)",
                  open(os.path.join(ROOT, "include", "gdn.h")).read())
    assert m and int(m.group(1)) * 1024 * 1024 == gdn.PREFILL_NOALLOC_SCRATCH_BYTES


def test_variant_and_layer_workspace_sizes():
    """gdn_prefill_variant_workspace_bytes adds, for a per-key decay with a decaying rule,
    the scaled Q and K (tokens x h_v x 128 16-bit values each, 1 KiB aligned);
    gdn_prefill_layer_workspace_bytes adds the convolved q, k (h_qk heads) and v (h_v
    heads) the same way.  Both are 0 off the tensor-core shapes."""
    up = lambda x: (x + 1023) // 1024 * 1024
    sh = gdn.make_shape(gdn.GDN_BF16, 2, 300, 2, 2, 4, 128, 128)
    base = gdn.gdn_prefill_workspace_bytes(sh)
    T = 600
    assert base > 0
    assert gdn.gdn_prefill_variant_workspace_bytes(sh) == base
    assert gdn.gdn_prefill_variant_workspace_bytes(sh, "delta", decay_per_key=True) == base
    assert gdn.gdn_prefill_variant_workspace_bytes(sh, "gated_delta", decay_per_key=True) == \
        base + 2 * up(T * 4 * 128 * 2)
    assert gdn.gdn_prefill_variant_workspace_bytes(sh, "gated", decay_per_key=True) == \
        base + 2 * up(T * 4 * 128 * 2)
    assert gdn.gdn_prefill_layer_workspace_bytes(sh) == \
        base + 2 * up(T * 2 * 128 * 2) + up(T * 4 * 128 * 2)
    off = gdn.make_shape(gdn.GDN_F32, 2, 300, 2, 2, 4, 128, 128)
    assert gdn.gdn_prefill_layer_workspace_bytes(off) == 0
    assert gdn.gdn_prefill_variant_workspace_bytes(off, "gated_delta", decay_per_key=True) == 0


def test_variant_plan_matches_the_prefill_plan():
    """Every rule, the shared beta and the per-key decay take gdn_prefill's path."""
    for sh in (gdn.make_shape(gdn.GDN_BF16, 1, 4096, 1, 16, 16, 128, 128),
               gdn.make_shape(gdn.GDN_F16, 1, 700, 3, 2, 4, 128, 128),
               gdn.make_shape(gdn.GDN_F32, 2, 64, 2, 2, 2, 32, 32)):
        want = gdn.gdn_prefill_plan(sh)
        for rule in gdn.RULES:
            for pk in (False, True):
                assert gdn.gdn_prefill_variant_plan(sh, rule, pk, False) == want
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_variant_plan(gdn.make_shape(gdn.GDN_BF16, 1, 64, 1, 1, 1, 128, 128), "nope")


def test_layer_prefill_rejects_bad_arguments_before_launch():
    lib = gdn.load()
    p = ctypes.c_void_p(0x1000)
    sh = gdn.make_shape(gdn.GDN_BF16, 1, 64, 1, 1, 1, 128, 128)

    def call(shape=sh, K=4, act=1, x=p, cs_in=p, cs_out=ctypes.c_void_p(0x80000)):
        layer = gdn.GdnLayerParams(K, act, gdn.ACTIVATIONS["silu"], 1e-6)
        return lib.gdn_prefill_layer(ctypes.byref(shape), ctypes.byref(layer), x, p, None, cs_in, cs_out,
                                     p, p, p, p, None, None, 0.0, p, p, ctypes.c_void_p(0x90000), p, 0,
                                     None, 0, None)

    assert call(K=5) == gdn.GDN_ERR_INVALID_ARG                     # more than 4 taps
    assert call(K=0) == gdn.GDN_ERR_INVALID_ARG
    assert call(act=2) == gdn.GDN_ERR_INVALID_ARG                   # sigmoid is not a conv activation
    assert call(x=ctypes.c_void_p(0x1008)) == gdn.GDN_ERR_INVALID_ARG   # x off 16 bytes
    assert call(cs_out=p) == gdn.GDN_ERR_INVALID_ARG                # the state updated in place
    assert call(cs_out=None) == gdn.GDN_ERR_INVALID_ARG
    f32 = gdn.make_shape(gdn.GDN_F32, 1, 64, 1, 1, 1, 128, 128)
    assert call(shape=f32) == gdn.GDN_ERR_UNSUPPORTED
