"""Pins for the CPU oracle: each test checks it against something other than itself.

CPU only (no GPU marker).  The pins come from the pages and from mathematics:
the worked example printed on the onnxruntime-ep-mlx ssm.rs page, closed forms
for special gates and rules, a retrieval invariant of the delta rule, a
brute-force product of per-token transition matrices, library routines for the
gate functions, and the float64 chunked re-association the GPU prefill uses.
"""
import json
import math
import os

import numpy as np
import pytest

import workloads
from chunked_ref import chunked_unit, chunked_unit_per_key

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_unit(rng, T, H, d):
    x = rng.standard_normal((T, H, d))
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- worked example

def test_worked_example_from_page(oracle_mod):
    """onnxruntime-ep-mlx ssm.rs unit test: linear rule, q = k = e0, v = 1/256."""
    import torch
    with open(os.path.join(GOLDEN, "linear_worked_example.json")) as f:
        fx = json.load(f)
    stored = fx["printed"]["state_bf16_after_T_steps"]
    for case in fx["cases"]:
        dk, T = case["d_k"], case["T"]
        q = np.zeros((T, 1, dk)); q[:, 0, 0] = 1.0
        v = np.full((T, 1, 1), 1.0 / 256.0)
        s0 = np.zeros((1, 1, dk, 1)); s0[0, 0, 0, 0] = 1.0
        o, s = oracle_mod.scan([0, T], 1, 1, dk, 1, q, q, v, state_in=s0, scale=1.0,
                               rule="linear")
        assert o.reshape(-1).tolist() == case["o"]              # exact, as printed
        # The page stores its state in bf16: round ours the same way.
        s_bf16 = torch.tensor(s.reshape(-1)).to(torch.bfloat16).to(torch.float64).numpy()
        assert s_bf16[0] == stored[str(T)]
        assert np.all(s_bf16[1:] == 0.0)
        assert s.reshape(-1)[0] == 1.0 + T / 256.0              # wide working state


# ---------------------------------------------------------------- gates

def test_gate_functions_against_library(oracle_mod):
    from scipy.special import expit
    xs = [-800.0, -50.0, -30.0, -3.5, -1.0, -1e-9, 0.0, 1e-9, 0.7, 2.0, 30.0, 50.0, 800.0]
    for x in xs:
        assert oracle_mod.sigmoid(x) == pytest.approx(float(expit(x)), rel=1e-15, abs=1e-300)
        assert oracle_mod.softplus(x) == pytest.approx(float(np.logaddexp(0.0, x)), rel=1e-15)
        # Identities: softplus(x) - softplus(-x) = x; sigmoid(x) + sigmoid(-x) = 1.
        assert oracle_mod.softplus(x) - oracle_mod.softplus(-x) == pytest.approx(x, abs=1e-12)
        assert oracle_mod.sigmoid(x) + oracle_mod.sigmoid(-x) == pytest.approx(1.0, abs=1e-15)
    assert oracle_mod.softplus(0.0) == math.log(2.0)
    assert oracle_mod.sigmoid(0.0) == 0.5
    assert oracle_mod.sigmoid(-math.inf) == 0.0 and oracle_mod.sigmoid(math.inf) == 1.0
    # g = -exp(A_log) softplus(a + dt_bias)
    assert oracle_mod.decay(0.0, 0.0, 0.0) == -math.log(2.0)
    assert oracle_mod.decay(0.25, math.log(3.0), -0.25) == pytest.approx(-3 * math.log(2.0), rel=1e-15)
    assert oracle_mod.decay(5.0, -math.inf, 1.0) == 0.0
    assert oracle_mod.decay(-60.0, 0.0, 0.0) == pytest.approx(-math.exp(-60.0), rel=1e-12)


def test_gates_end_to_end_half_decay_and_half_beta(oracle_mod):
    """A_log = 0, a + dt_bias = 0 gives alpha = 1/2; b = 0 gives beta = 1/2."""
    rng = np.random.default_rng(1)
    dk, dv = 8, 5
    q = _rand_unit(rng, 1, 1, dk)
    s0 = rng.standard_normal((1, 1, dk, dv))
    # k = 0: nothing is written, so S1 = alpha S0 and o = scale alpha S0^T q.
    o, s = oracle_mod.scan([0, 1], 1, 1, dk, dv, q, np.zeros((1, 1, dk)),
                           rng.standard_normal((1, 1, dv)), a=[0.3], b=[0.0], A_log=[0.0],
                           dt_bias=[-0.3], state_in=s0, scale=1.0)
    assert _rel(s, 0.5 * s0) < 1e-15
    assert _rel(o[0, 0], 0.5 * (s0[0, 0].T @ q[0, 0])) < 1e-14
    # From zero state with alpha irrelevant: S = beta k v^T, o = beta (q.k) v.
    k = _rand_unit(rng, 1, 1, dk)
    v = rng.standard_normal((1, 1, dv))
    o, s = oracle_mod.scan([0, 1], 1, 1, dk, dv, q, k, v, a=[0.0], b=[0.0], A_log=[0.0],
                           dt_bias=[0.0], scale=1.0)
    assert _rel(s[0, 0], 0.5 * np.outer(k[0, 0], v[0, 0])) < 1e-15
    assert _rel(o[0, 0], 0.5 * (q[0, 0] @ k[0, 0]) * v[0, 0]) < 1e-14


# ---------------------------------------------------------------- invariants

def test_invariant_a_no_gate_no_write(oracle_mod):
    """beta = 0 and g = 0 (b = -inf, A_log = -inf): from a zero state o = 0 and S = 0;
    from any state, S is unchanged and o_t = scale S0^T q_t."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 6, 2, 16, 12
    q, k = _rand_unit(rng, T, H, dk), _rand_unit(rng, T, H, dk)
    v = rng.standard_normal((T, H, dv))
    a = rng.standard_normal((T, H))
    b = np.full((T, H), -np.inf)
    A_log = np.full(H, -np.inf)
    dt = rng.normal(0, 0.1, H)
    o, s = oracle_mod.scan([0, T], H, H, dk, dv, q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt)
    assert np.all(o == 0.0) and np.all(s == 0.0)
    s0 = rng.standard_normal((1, H, dk, dv))
    o, s = oracle_mod.scan([0, T], H, H, dk, dv, q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt,
                           state_in=s0, scale=0.5)
    assert np.array_equal(s, s0)
    for t in range(T):
        for h in range(H):
            assert _rel(o[t, h], 0.5 * s0[0, h].T @ q[t, h]) < 1e-14


def test_invariant_b_linear_rule_is_causal_linear_attention(oracle_mod):
    """Rule linear with g = 0: o_t = scale sum_{s<=t} (q_t.k_s) v_s (direct O(T^2) sum)."""
    rng = np.random.default_rng(3)
    T, H, dk, dv = 40, 2, 16, 24
    q, k = rng.standard_normal((T, H, dk)), rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    o, s = oracle_mod.scan([0, T], H, H, dk, dv, q, k, v, scale=0.3, rule="linear")
    for h in range(H):
        for t in range(T):
            ref = 0.3 * sum((q[t, h] @ k[s_, h]) * v[s_, h] for s_ in range(t + 1))
            assert _rel(o[t, h], ref) < 1e-12
        assert _rel(s[0, h], sum(np.outer(k[s_, h], v[s_, h]) for s_ in range(T))) < 1e-12


def test_gated_rule_is_decayed_linear_attention(oracle_mod):
    """Rule gated: o_t = scale (e^{G_t} S0^T q_t + sum_{s<=t} e^{G_t-G_s} (q_t.k_s) v_s)."""
    rng = np.random.default_rng(4)
    T, dk, dv = 30, 8, 6
    q, k = rng.standard_normal((T, 1, dk)), rng.standard_normal((T, 1, dk))
    v = rng.standard_normal((T, 1, dv))
    g = -rng.uniform(0, 0.5, (T, 1))
    s0 = rng.standard_normal((1, 1, dk, dv))
    o, _ = oracle_mod.scan([0, T], 1, 1, dk, dv, q, k, v, g=g, state_in=s0, scale=1.0,
                           rule="gated")
    G = np.cumsum(g[:, 0])
    for t in range(T):
        ref = np.exp(G[t]) * s0[0, 0].T @ q[t, 0]
        ref = ref + sum(np.exp(G[t] - G[s_]) * (q[t, 0] @ k[s_, 0]) * v[s_, 0]
                        for s_ in range(t + 1))
        assert _rel(o[t, 0], ref) < 1e-12


def test_invariant_c_delta_rule_retrieval(oracle_mod):
    """beta = 1, unit keys, g = 0: after writing (k1,v1), (k2 _|_ k1, v2), (k1,v3),
    reading with k1 returns v3 and reading with k2 returns v2."""
    rng = np.random.default_rng(5)
    dk, dv = 16, 10
    k1 = rng.standard_normal(dk); k1 /= np.linalg.norm(k1)
    k2 = rng.standard_normal(dk); k2 -= (k2 @ k1) * k1; k2 /= np.linalg.norm(k2)
    v1, v2, v3 = rng.standard_normal((3, dv))
    ks = np.stack([k1, k2, k1, k1, k2])[:, None, :]
    vs = np.stack([v1, v2, v3, np.zeros(dv), np.zeros(dv)])[:, None, :]
    # Tokens 4 and 5 read with q = k1, k2; beta = 0 there so they write nothing.
    qs = ks.copy()
    b = np.array([np.inf, np.inf, np.inf, -np.inf, -np.inf])[:, None]
    o, s = oracle_mod.scan([0, 5], 1, 1, dk, dv, qs, ks, vs, a=np.zeros((5, 1)), b=b,
                           A_log=[-np.inf], dt_bias=[0.0], scale=1.0)
    assert np.max(np.abs(o[3, 0] - v3)) < 1e-14
    assert np.max(np.abs(o[4, 0] - v2)) < 1e-14
    assert np.max(np.abs(o[2, 0] - v3)) < 1e-14     # readout uses the updated state
    assert np.max(np.abs(s[0, 0].T @ k1 - v3)) < 1e-14


def _transition_bruteforce(q, k, v, g, beta, S0, scale):
    """S_t = A_t ... A_1 S0 + sum_s A_t ... A_{s+1} beta_s k_s v_s^T with
    A_t = e^{g_t} (I - beta_t k_t k_t^T); o_t = scale S_t^T q_t."""
    T, dk = k.shape
    A = [np.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])) for t in range(T)]

    def phi(t, s):          # A_t A_{t-1} ... A_{s+1}  (0-based t, s exclusive)
        M = np.eye(dk)
        for r in range(s + 1, t + 1):
            M = A[r] @ M
        return M

    o = []
    S = None
    for t in range(T):
        S = phi(t, -1) @ S0
        for s in range(t + 1):
            S = S + phi(t, s) @ (beta[s] * np.outer(k[s], v[s]))
        o.append(scale * S.T @ q[t])
    return np.array(o), S


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_invariant_d_bruteforce(oracle_mod, T):
    """Random gates, GQA (2 value heads per q/k head), d_k != d_v, a nonzero state."""
    rng = np.random.default_rng(10 + T)
    h_qk, h_v, dk, dv = 2, 4, 6, 5
    q, k = _rand_unit(rng, T, h_qk, dk), _rand_unit(rng, T, h_qk, dk)
    v = rng.standard_normal((T, h_v, dv))
    g = -rng.uniform(0.0, 1.5, (T, h_v))
    beta = rng.uniform(0.0, 1.0, (T, h_v))
    s0 = rng.standard_normal((1, h_v, dk, dv))
    o, s = oracle_mod.scan([0, T], h_qk, h_v, dk, dv, q, k, v, g=g, beta=beta, state_in=s0,
                           scale=0.7)
    for h in range(h_v):
        hq = h // (h_v // h_qk)
        ob, sb = _transition_bruteforce(q[:, hq], k[:, hq], v[:, h], g[:, h], beta[:, h],
                                        s0[0, h], 0.7)
        assert _rel(o[:, h], ob) < 1e-12
        assert _rel(s[0, h], sb) < 1e-12


def test_delta_rule_equals_gated_delta_with_zero_decay(oracle_mod):
    rng = np.random.default_rng(6)
    T, dk, dv = 12, 8, 8
    q, k = _rand_unit(rng, T, 1, dk), _rand_unit(rng, T, 1, dk)
    v = rng.standard_normal((T, 1, dv))
    beta = rng.uniform(0, 1, (T, 1))
    o1, s1 = oracle_mod.scan([0, T], 1, 1, dk, dv, q, k, v, beta=beta, rule="delta",
                             g=-np.ones((T, 1)))
    o2, s2 = oracle_mod.scan([0, T], 1, 1, dk, dv, q, k, v, beta=beta, g=np.zeros((T, 1)))
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


# ---------------------------------------------------------------- composition, edges

def test_composition_chaining_varlen_and_gqa(oracle_mod):
    spec = workloads.small_spec(io="bf16", lengths=[37, 0, 64, 101], h_qk=2, h_v=4, d_k=16,
                                d_v=8, seed=21, state_std=0.05)
    inp = workloads.draw(spec)
    o, s = oracle_mod.scan_inputs(inp)
    f = inp.f64
    cu = inp.cu_seqlens
    hq, hv, dk, dv = spec.h_qk, spec.h_v, spec.d_k, spec.d_v
    q, k = f["q"].reshape(-1, hq, dk), f["k"].reshape(-1, hq, dk)
    v = f["v"].reshape(-1, hv, dv)
    a, b = f["a"].reshape(-1, hv), f["b"].reshape(-1, hv)
    s0 = f["state_in"].reshape(-1, hv, dk, dv)
    kw = dict(A_log=f["A_log"], dt_bias=f["dt_bias"], scale=inp.scale)
    for n in range(len(cu) - 1):
        t0, t1 = cu[n], cu[n + 1]
        sl = slice(t0, t1)
        # varlen == one call per sequence (bit-identical)
        o1, s1 = oracle_mod.scan([0, t1 - t0], hq, hv, dk, dv, q[sl], k[sl], v[sl], a=a[sl],
                                 b=b[sl], state_in=s0[n:n + 1], **kw)
        assert np.array_equal(o1, o[sl]) and np.array_equal(s1[0], s[n])
        # chaining: run the first part, then the rest from its state
        m = t0 + (t1 - t0) // 3
        oa, sa = oracle_mod.scan([0, m - t0], hq, hv, dk, dv, q[t0:m], k[t0:m], v[t0:m],
                                 a=a[t0:m], b=b[t0:m], state_in=s0[n:n + 1], **kw)
        ob, sb = oracle_mod.scan([0, t1 - m], hq, hv, dk, dv, q[m:t1], k[m:t1], v[m:t1],
                                 a=a[m:t1], b=b[m:t1], state_in=sa, **kw)
        assert np.array_equal(np.concatenate([oa, ob]), o[sl]) and np.array_equal(sb[0], s[n])
    # GQA == the same call with each q/k head repeated for its value heads
    rep = hv // hq
    o2, s2 = oracle_mod.scan(cu, hv, hv, dk, dv, np.repeat(q, rep, axis=1),
                             np.repeat(k, rep, axis=1), v, a=a, b=b, state_in=s0, **kw)
    assert np.array_equal(o2, o) and np.array_equal(s2, s)
    # A unit subset computes exactly those units
    units = [1, 6, 13]
    o3, s3 = oracle_mod.scan_inputs(inp, units=units)
    for u in units:
        n, h = divmod(u, hv)
        assert np.array_equal(s3[n, h], s[n, h])
        assert np.array_equal(o3[cu[n]:cu[n + 1], h], o[cu[n]:cu[n + 1], h])


def test_empty_time_axis_keeps_state(oracle_mod):
    rng = np.random.default_rng(8)
    s0 = rng.standard_normal((2, 3, 4, 5))
    e = np.zeros((0,))
    o, s = oracle_mod.scan([0, 0, 0], 3, 3, 4, 5, e, e, e, a=e, b=e, A_log=np.zeros(3),
                           dt_bias=np.zeros(3), state_in=s0)
    assert o.shape == (0, 3, 5) and np.array_equal(s, s0)
    o, s = oracle_mod.scan([0, 0], 3, 3, 4, 5, e, e, e, a=e, b=e, A_log=np.zeros(3),
                           dt_bias=np.zeros(3))
    assert np.all(s == 0.0)


def test_threads_do_not_change_results(oracle_mod):
    inp = workloads.draw(workloads.small_spec(lengths=[50, 70, 3], h_qk=2, h_v=2, d_k=16,
                                              d_v=16, seed=9))
    o1, s1 = oracle_mod.scan_inputs(inp, threads=1)
    o2, s2 = oracle_mod.scan_inputs(inp, threads=4)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


# ---------------------------------------------------------------- the chunked algebra

@pytest.mark.parametrize("C,L", [(64, 64), (64, 200), (16, 37), (64, 1), (32, 128)])
def test_chunked_reassociation_matches_sequential(oracle_mod, C, L):
    """The WY/UT chunked form the GPU prefill uses equals the recurrence in float64."""
    spec = workloads.small_spec(io="f32", lengths=[L], h_qk=1, h_v=2, d_k=32, d_v=16,
                                seed=100 + L, state_std=0.05)
    inp = workloads.draw(spec)
    o, s = oracle_mod.scan_inputs(inp)
    f = inp.f64
    q, k = f["q"].reshape(L, 1, 32), f["k"].reshape(L, 1, 32)
    v = f["v"].reshape(L, 2, 16)
    for h in range(2):
        g = np.array([oracle_mod.decay(x, f["A_log"][h], f["dt_bias"][h])
                      for x in f["a"].reshape(L, 2)[:, h]])
        beta = np.array([oracle_mod.sigmoid(x) for x in f["b"].reshape(L, 2)[:, h]])
        oc, sc = chunked_unit(q[:, 0], k[:, 0], v[:, h], g, beta,
                              f["state_in"].reshape(1, 2, 32, 16)[0, h], inp.scale, C)
        assert _rel(oc, o[:, h]) < 1e-11
        assert _rel(sc, s[0, h]) < 1e-11


@pytest.mark.parametrize("C,L,bump", [(64, 200, 0.0), (16, 37, 0.0), (64, 64, 3.0), (32, 100, 3.0)])
def test_chunked_per_key_reassociation_matches_sequential(oracle_mod, C, L, bump):
    """The per-key-dimension chunked form the GPU prefill uses (gates inside A, P, W, the
    scaled Q and K and the per-row carry) equals the recurrence in float64; bump raises
    A_log on every other key dimension so those decay up to ~160 per token."""
    spec = workloads.small_spec(io="f32", lengths=[L], h_qk=1, h_v=2, d_k=32, d_v=16,
                                seed=200 + L, state_std=0.05, decay_per_key=True)
    inp = workloads.draw(spec)
    f = dict(inp.f64)
    A_log = f["A_log"].reshape(2, 32).copy()
    A_log[:, 1::2] += bump
    f["A_log"] = A_log.reshape(-1)
    o, s = oracle_mod.scan(inp.cu_seqlens, 1, 2, 32, 16, f["q"], f["k"], f["v"], a=f["a"],
                           b=f["b"], A_log=f["A_log"], dt_bias=f["dt_bias"],
                           state_in=f["state_in"], scale=inp.scale, decay_per_key=True)
    q, k = f["q"].reshape(L, 1, 32), f["k"].reshape(L, 1, 32)
    v = f["v"].reshape(L, 2, 16)
    a = f["a"].reshape(L, 2, 32)
    dtb = f["dt_bias"].reshape(2, 32)
    for h in range(2):
        g = np.array([[oracle_mod.decay(a[t, h, i], A_log[h, i], dtb[h, i]) for i in range(32)]
                      for t in range(L)])
        beta = np.array([oracle_mod.sigmoid(x) for x in f["b"].reshape(L, 2)[:, h]])
        oc, sc = chunked_unit_per_key(q[:, 0], k[:, 0], v[:, h], g, beta,
                                      f["state_in"].reshape(1, 2, 32, 16)[0, h], inp.scale, C)
        assert _rel(oc, o[:, h]) < 1e-11
        assert _rel(sc, s[0, h]) < 1e-11


def test_workload_recipe():
    """The measured workloads' shapes and draws (c3's lengths are drawn first); the
    slot-pool decode workload names distinct pool entries."""
    w = workloads.WORKLOADS
    assert set(w) == {"tiny_f32_prefill", "bf16_prefill_t4096", "bf16_decode_b256",
                      "varlen_bf16_prefill", "gqa_f16_prefill", "bf16_slot_decode_b256",
                      "bf16_window_b256_t4", "bf16_perkey_decode_b256", "bf16_delta_prefill_t4096",
                      "bf16_shared_beta_prefill_t4096", "bf16_perkey_prefill_t4096"}
    assert w["bf16_delta_prefill_t4096"].rule == "delta"
    assert all(w[n].rule == "gated_delta" for n in w if n != "bf16_delta_prefill_t4096")
    assert set(workloads.CONV_WORKLOADS) == {"bf16_conv_prefill_gqa", "bf16_conv_decode_b256"}
    assert set(workloads.NORM_WORKLOADS) == {"bf16_norm_gqa"}
    cv = workloads.draw_conv(workloads.ConvSpec("t", "bf16", 2, 5, 8, 3, state_std=1.0,
                                                state_window=2, bias=True))
    assert tuple(cv.x.shape) == (2, 5, 8) and tuple(cv.w.shape) == (8, 1, 4)
    assert tuple(cv.state_in.shape) == (2, 2, 3, 8) and tuple(cv.bias.shape) == (8,)
    assert float(cv.w.abs().max()) <= 0.5        # U(-1/sqrt(K), 1/sqrt(K)), K = 4
    pool = workloads.draw_conv(workloads.ConvSpec("t", "bf16", 3, 1, 8, 4, state_std=1.0,
                                                  pool_size=6))
    assert len(set(pool.slots.tolist())) == 3 and tuple(pool.pool.shape) == (6, 3, 8)
    nm = workloads.draw_norm(workloads.NormSpec("n", "f16", (2, 3, 16), 5))
    assert tuple(nm.x.shape) == tuple(nm.gate.shape) == (2, 3, 16) and tuple(nm.scale.shape) == (16,)
    pk = workloads.draw(workloads.small_spec(io="bf16", batch=3, seqlen=2, h_qk=1, h_v=2, d_k=8,
                                             d_v=4, decay_per_key=True, beta_shared=True))
    assert tuple(pk.a.shape) == (3, 2, 2, 8) and tuple(pk.A_log.shape) == (2, 8)
    assert tuple(pk.dt_bias.shape) == (2, 8) and tuple(pk.b.shape) == (3, 2, 1)
    sp = w["bf16_slot_decode_b256"]
    sl = workloads.draw(workloads.small_spec(io="bf16", batch=sp.batch, seqlen=1, h_qk=1, h_v=1,
                                             d_k=4, d_v=4, decode=True, pool_size=sp.pool_size,
                                             pool_std=0.05, seed=sp.seed)).slots.numpy()
    assert len(set(sl.tolist())) == sp.batch and sl.min() >= 0 and sl.max() < sp.pool_size
    rng = np.random.default_rng(1003)
    lengths = rng.integers(512, 8193, 8)
    assert np.all((lengths >= 512) & (lengths <= 8192))
    inp = workloads.draw(workloads.small_spec(io="bf16", lengths=[3, 4], h_qk=1, h_v=1,
                                              d_k=64, d_v=8))
    qn = np.linalg.norm(inp.f64["q"].reshape(-1, 64), axis=-1)
    assert np.all(np.abs(qn - 1.0) < 1e-2)   # unit norm up to the bf16 cast


# ---------------------------------------------------------------- state pool (slots)

def _pool_case(n=5, pool_size=9, seqlen=1, seed=3):
    return workloads.draw(workloads.small_spec(io="f32", batch=n, seqlen=seqlen, h_qk=1, h_v=2,
                                               d_k=16, d_v=8, decode=(seqlen == 1),
                                               pool_size=pool_size, pool_std=0.05, seed=seed))


def test_slot_scan_with_identity_slots_is_the_plain_scan(oracle_mod):
    """take(pool, arange(n)) is the pool itself, so the slot op must equal the plain op
    started from the pool (nuvec-core gated_delta_slots fallback: take, rule, put)."""
    inp = _pool_case(n=4, pool_size=4)
    f, s = inp.f64, inp.spec
    o, pool = oracle_mod.slot_scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"],
                               f["v"], f["a"], f["b"], f["A_log"], f["dt_bias"], f["pool"],
                               np.arange(4), scale=inp.scale)
    o_ref, s_ref = oracle_mod.scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"],
                               f["v"], a=f["a"], b=f["b"], A_log=f["A_log"],
                               dt_bias=f["dt_bias"], state_in=f["pool"], scale=inp.scale)
    assert np.array_equal(o, o_ref) and np.array_equal(pool, s_ref)


def test_slot_scan_leaves_unnamed_entries_and_commutes_with_a_pool_permutation(oracle_mod):
    inp = _pool_case()
    f, s = inp.f64, inp.spec
    slots = inp.slots.numpy()
    args = (inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"], f["v"], f["a"],
            f["b"], f["A_log"], f["dt_bias"])
    pool0 = f["pool"].reshape(9, s.h_v, s.d_k, s.d_v)
    o, pool = oracle_mod.slot_scan(*args, pool0, slots, scale=inp.scale)
    untouched = sorted(set(range(9)) - set(int(x) for x in slots))
    assert untouched and np.array_equal(pool[untouched], pool0[untouched])
    for x in slots:
        assert not np.array_equal(pool[x], pool0[x])
    # Relabel the pool entries with a permutation pi: entry e moves to pi[e].
    pi = np.random.default_rng(5).permutation(9)
    pool_p = np.empty_like(pool0)
    pool_p[pi] = pool0
    o_p, pool_pp = oracle_mod.slot_scan(*args, pool_p, pi[slots], scale=inp.scale)
    assert np.array_equal(o_p, o)
    assert np.array_equal(pool_pp[pi], pool)


def test_slot_scan_skips_a_slot_outside_the_pool(oracle_mod):
    inp = _pool_case()
    f, s = inp.f64, inp.spec
    slots = inp.slots.numpy().copy()
    slots[2] = 9                                  # one past the end
    o, pool = oracle_mod.slot_scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"],
                               f["v"], f["a"], f["b"], f["A_log"], f["dt_bias"], f["pool"],
                               slots, scale=inp.scale)
    pool0 = f["pool"].reshape(9, s.h_v, s.d_k, s.d_v)
    assert np.all(o[2] == 0.0)
    kept = [int(x) for i, x in enumerate(slots) if i != 2]
    others = sorted(set(range(9)) - set(kept))
    assert np.array_equal(pool[others], pool0[others])


def test_slot_scan_over_several_steps_equals_single_steps(oracle_mod):
    """The page's op runs T steps per row; T = 3 must equal three T = 1 slot steps that
    each pick up the pool the previous one left (composition)."""
    inp = _pool_case(n=3, pool_size=6, seqlen=3, seed=8)
    f, s = inp.f64, inp.spec
    slots = inp.slots.numpy()
    o3, pool3 = oracle_mod.slot_scan(inp.cu_seqlens, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"],
                                 f["v"], f["a"], f["b"], f["A_log"], f["dt_bias"], f["pool"],
                                 slots, scale=inp.scale)
    q = f["q"].reshape(3, 3, s.h_qk, s.d_k)
    k = f["k"].reshape(3, 3, s.h_qk, s.d_k)
    v = f["v"].reshape(3, 3, s.h_v, s.d_v)
    a = f["a"].reshape(3, 3, s.h_v)
    b = f["b"].reshape(3, 3, s.h_v)
    pool = f["pool"]
    cu1 = np.arange(4)
    for t in range(3):
        o1, pool = oracle_mod.slot_scan(cu1, s.h_qk, s.h_v, s.d_k, s.d_v, q[:, t], k[:, t], v[:, t],
                                    a[:, t], b[:, t], f["A_log"], f["dt_bias"], pool, slots,
                                    scale=inp.scale)
        assert np.allclose(o1, o3.reshape(3, 3, s.h_v, s.d_v)[:, t], rtol=1e-12, atol=1e-14)
    assert np.allclose(pool, pool3, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- state window

def _window_case(B=2, T=5, seed=9):
    return workloads.draw(workloads.small_spec(io="f32", batch=B, seqlen=T, h_qk=1, h_v=2,
                                               d_k=16, d_v=8, state_std=0.05, seed=seed))


def _window(oracle_mod, inp, W):
    s, f = inp.spec, inp.f64
    return oracle_mod.window_scan(s.batch, s.seqlen, s.h_qk, s.h_v, s.d_k, s.d_v, f["q"], f["k"],
                                  f["v"], f["a"], f["b"], f["A_log"], f["dt_bias"],
                                  f["state_in"], W, scale=inp.scale)


def test_window_last_slab_is_the_final_state_and_outputs_agree(oracle_mod):
    inp = _window_case()
    o_ref, s_ref = oracle_mod.scan_inputs(inp)
    o, win = _window(oracle_mod, inp, 1)
    assert np.array_equal(win[0], s_ref)
    assert np.array_equal(o, o_ref.reshape(o.shape))


def test_window_slabs_are_the_states_of_shorter_runs(oracle_mod):
    """window[W-1-j] is the final state of the same run stopped j steps early."""
    inp = _window_case(T=6)
    o, win = _window(oracle_mod, inp, 4)
    s, f = inp.spec, inp.f64
    for j in range(4):
        L = s.seqlen - j
        sub = lambda x, last: x.reshape(s.batch, s.seqlen, *last)[:, :L].reshape(-1)
        _, s_short = oracle_mod.scan(np.arange(s.batch + 1) * L, s.h_qk, s.h_v, s.d_k, s.d_v,
                                     sub(f["q"], (s.h_qk, s.d_k)), sub(f["k"], (s.h_qk, s.d_k)),
                                     sub(f["v"], (s.h_v, s.d_v)), a=sub(f["a"], (s.h_v,)),
                                     b=sub(f["b"], (s.h_v,)), A_log=f["A_log"],
                                     dt_bias=f["dt_bias"], state_in=f["state_in"], scale=inp.scale)
        assert np.allclose(win[3 - j], s_short, rtol=1e-12, atol=1e-15)


def test_window_longer_than_the_run_starts_with_zero_slabs(oracle_mod):
    inp = _window_case(T=3)
    _, win = _window(oracle_mod, inp, 5)
    assert np.all(win[:2] == 0.0)
    _, s_ref = oracle_mod.scan_inputs(inp)
    assert np.array_equal(win[4], s_ref)
    assert np.all(np.any(win[2:] != 0.0, axis=(1, 2, 3, 4)))


# ---------------------------------------------------------------- gate and rule variants

def _variant_case(T=7, h_v=2, d_k=6, d_v=4, seed=21):
    rng = np.random.default_rng(seed)
    q = _rand_unit(rng, T, 1, d_k)
    k = _rand_unit(rng, T, 1, d_k)
    v = rng.standard_normal((T, h_v, d_v))
    return rng, q, k, v


def test_per_key_decay_with_equal_factors_is_the_per_head_decay(oracle_mod):
    rng, q, k, v = _variant_case()
    T, h_v, d_k, d_v = 7, 2, 6, 4
    a = rng.standard_normal((T, h_v))
    b = rng.standard_normal((T, h_v))
    A_log = rng.uniform(-1, 1, h_v)
    dt = rng.normal(0, 0.1, h_v)
    cu = [0, T]
    o1, s1 = oracle_mod.scan(cu, 1, h_v, d_k, d_v, q, k, v, a=a, b=b, A_log=A_log, dt_bias=dt)
    rep = lambda x: np.repeat(x[..., None], d_k, axis=-1)
    o2, s2 = oracle_mod.scan(cu, 1, h_v, d_k, d_v, q, k, v, a=rep(a), b=b, A_log=rep(A_log),
                             dt_bias=rep(dt), decay_per_key=True)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_per_key_decay_gated_rule_closed_form(oracle_mod):
    """Rule `gated` with one decay per key dimension from a zero state:
    S_t = sum_{s<=t} diag(prod_{r=s+1..t} alpha_r) k_s v_s^T, o_t = scale S_t^T q_t."""
    rng, q, k, v = _variant_case()
    T, h_v, d_k, d_v = 7, 2, 6, 4
    g = -rng.uniform(0.0, 0.7, (T, h_v, d_k))
    scale = 0.37
    o, s = oracle_mod.scan([0, T], 1, h_v, d_k, d_v, q, k, v, g=g, scale=scale, rule="gated",
                           decay_per_key=True)
    alpha = np.exp(g)
    for h in range(h_v):
        for t in range(T):
            St = np.zeros((d_k, d_v))
            for s_ in range(t + 1):
                f = np.prod(alpha[s_ + 1:t + 1, h, :], axis=0)
                St += np.outer(f * k[s_, 0], v[s_, h])
            assert _rel(o[t, h], scale * St.T @ q[t, 0]) < 1e-12
        assert _rel(s[0, h], St) < 1e-12


def test_shared_beta_equals_the_replicated_per_head_beta(oracle_mod):
    rng, q, k, v = _variant_case()
    T, h_v, d_k, d_v = 7, 2, 6, 4
    a = rng.standard_normal((T, h_v))
    b1 = rng.standard_normal(T)
    A_log = rng.uniform(-1, 1, h_v)
    dt = rng.normal(0, 0.1, h_v)
    o1, s1 = oracle_mod.scan([0, T], 1, h_v, d_k, d_v, q, k, v, a=a, b=b1, A_log=A_log,
                             dt_bias=dt, beta_shared=True)
    o2, s2 = oracle_mod.scan([0, T], 1, h_v, d_k, d_v, q, k, v, a=a,
                             b=np.repeat(b1[:, None], h_v, axis=1), A_log=A_log, dt_bias=dt)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_delta_rule_is_gated_delta_without_decay(oracle_mod):
    rng, q, k, v = _variant_case()
    T, h_v, d_k, d_v = 7, 2, 6, 4
    beta = rng.uniform(0, 1, (T, h_v))
    s0 = rng.normal(0, 0.1, (1, h_v, d_k, d_v))
    o1, s1 = oracle_mod.scan([0, T], 1, h_v, d_k, d_v, q, k, v, beta=beta, state_in=s0,
                             rule="delta")
    o2, s2 = oracle_mod.scan([0, T], 1, h_v, d_k, d_v, q, k, v, g=np.zeros((T, h_v)),
                             beta=beta, state_in=s0, rule="gated_delta")
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


@pytest.mark.parametrize("m", [1, 17, 39])
def test_time_parallel_decomposition(oracle_mod, m):
    """The recurrence is linear in the state, which the time-parallel prefill relies on.
    Cut a sequence after token m, with S_m the state there:
      - the run from S_m equals the run from zero plus the run with v = 0 from S_m;
      - the run with v = 0 from S_m equals, column by column, the run with v = 0 from the
        identity (the operator pass, d_v = d_k) times S_m;
    so o_t = o0_t + R_t S_m and S_end = Phi S_m + Psi, with R, Phi from the operator pass."""
    rng = np.random.default_rng(70 + m)
    T, hq, hv, dk, dv = 40, 1, 2, 8, 6
    q = rng.standard_normal((T, hq, dk))
    k = rng.standard_normal((T, hq, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, hv, dv))
    a, b = rng.standard_normal((T, hv)), rng.standard_normal((T, hv))
    A_log, dt = rng.uniform(-1, 1, hv), rng.normal(0, 0.1, hv)
    s0 = rng.normal(0, 0.1, (1, hv, dk, dv))
    gates = lambda sl: dict(a=a[sl], b=b[sl], A_log=A_log, dt_bias=dt)
    full_o, full_s = oracle_mod.scan([0, T], hq, hv, dk, dv, q, k, v, state_in=s0, **gates(slice(None)))
    _, s_m = oracle_mod.scan([0, m], hq, hv, dk, dv, q[:m], k[:m], v[:m], state_in=s0,
                             **gates(slice(0, m)))
    rest = slice(m, T)
    o0, psi = oracle_mod.scan([0, T - m], hq, hv, dk, dv, q[rest], k[rest], v[rest], **gates(rest))
    eye = np.broadcast_to(np.eye(dk), (1, hv, dk, dk)).copy()
    R, phi = oracle_mod.scan([0, T - m], hq, hv, dk, dk, q[rest], k[rest],
                             np.zeros((T - m, hv, dk)), state_in=eye, **gates(rest))
    for h in range(hv):
        o_pred = o0[:, h] + R[:, h] @ s_m[0, h]
        assert _rel(o_pred, full_o[m:, h]) < 1e-12
        assert _rel(phi[0, h] @ s_m[0, h] + psi[0, h], full_s[0, h]) < 1e-12
