"""Pins of the oracle's neighbouring ops: CausalConvWithState and GatedRMSNorm.

Each check rests on something other than the oracle's own loops: numpy's correlate,
the impulse response, composition of calls, algebraic identities of silu and of the
RMS normalisation, and closed forms.  No GPU needed."""
import numpy as np
import pytest


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    d = np.max(np.abs(a - b)) if a.size else 0.0
    m = np.max(np.abs(b)) if b.size else 0.0
    return d / m if m > 0 else d


def _case(rng, B=2, L=11, C=5, K=4, dil=1):
    carry = (K - 1) * dil
    x = rng.standard_normal((B, L, C))
    w = rng.standard_normal((C, 1, K))
    bias = rng.standard_normal(C)
    st = rng.standard_normal((B, carry, C))
    return x, w, bias, st


# ------------------------------------------------------------------ causal conv

@pytest.mark.parametrize("K,dil", [(1, 1), (3, 1), (4, 1), (4, 2), (2, 5)])
def test_conv_is_numpy_correlate_over_the_padded_sequence(oracle_mod, K, dil):
    rng = np.random.default_rng(40 + K + dil)
    x, w, bias, st = _case(rng, K=K, dil=dil)
    y, _ = oracle_mod.causal_conv(x, w, bias, st, dilation=dil)
    B, L, C = x.shape
    for b in range(B):
        for c in range(C):
            padded = np.concatenate([st[b, :, c], x[b, :, c]])
            taps = np.zeros((K - 1) * dil + 1)
            taps[::dil] = w[c, 0]
            ref = np.correlate(padded, taps, mode="valid") + bias[c]
            assert _rel(y[b, :, c], ref) < 1e-13


def test_conv_impulse_response_is_the_reversed_kernel(oracle_mod):
    """A unit impulse at t0 with a zero state: y[t0 + m * dil] = w[K - 1 - m]."""
    K, dil, L, t0 = 4, 3, 20, 2
    w = np.arange(1.0, K + 1).reshape(1, 1, K)
    x = np.zeros((1, L, 1))
    x[0, t0, 0] = 1.0
    y, _ = oracle_mod.causal_conv(x, w, dilation=dil)
    want = np.zeros(L)
    for m in range(K):
        want[t0 + m * dil] = w[0, 0, K - 1 - m]
    assert np.array_equal(y[0, :, 0], want)


@pytest.mark.parametrize("split", [0, 1, 2, 7, 11])
def test_conv_chained_calls_equal_one_call(oracle_mod, split):
    rng = np.random.default_rng(7)
    x, w, bias, st = _case(rng, L=11, K=4, dil=2)
    y, s = oracle_mod.causal_conv(x, w, bias, st, dilation=2, silu=True)
    y1, s1 = oracle_mod.causal_conv(x[:, :split], w, bias, st, dilation=2, silu=True)
    y2, s2 = oracle_mod.causal_conv(x[:, split:], w, bias, s1, dilation=2, silu=True)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(s2, s)


def test_conv_state_is_the_last_padded_positions(oracle_mod):
    rng = np.random.default_rng(8)
    x, w, bias, st = _case(rng, L=9, K=5)            # carry 4 <= L
    _, s = oracle_mod.causal_conv(x, w, bias, st)
    assert np.array_equal(s, x[:, -4:])
    _, s = oracle_mod.causal_conv(x[:, :2], w, bias, st)   # L = 2 < carry: 2 old, 2 new
    assert np.array_equal(s, np.concatenate([st[:, 2:], x[:, :2]], axis=1))
    _, s = oracle_mod.causal_conv(x[:, :0], w, bias, st)   # no token: unchanged
    assert np.array_equal(s, st)
    _, s = oracle_mod.causal_conv(x[:, :2], w, bias, None)  # no past state: zeros first
    assert np.array_equal(s[:, :2], np.zeros_like(s[:, :2]))


def test_conv_silu_odd_part_is_the_plain_convolution(oracle_mod):
    """silu(p) - silu(-p) = p: negating the taps and the bias negates p."""
    rng = np.random.default_rng(9)
    x, w, bias, st = _case(rng)
    yp, _ = oracle_mod.causal_conv(x, w, bias, st, silu=True)
    ym, _ = oracle_mod.causal_conv(x, -w, -bias, st, silu=True)
    y0, _ = oracle_mod.causal_conv(x, w, bias, st)
    assert _rel(yp - ym, y0) < 1e-14
    assert np.all(yp >= -0.2785)   # silu's minimum is about -0.27846


def test_conv_channel_layouts_agree(oracle_mod):
    rng = np.random.default_rng(10)
    x, w, bias, st = _case(rng, K=3, dil=2)
    y, s = oracle_mod.causal_conv(x, w, bias, st, dilation=2, silu=True)
    yf, sf = oracle_mod.causal_conv(x.transpose(0, 2, 1), w, bias, st.transpose(0, 2, 1),
                                    dilation=2, silu=True, channels_last=False)
    assert np.array_equal(yf, y.transpose(0, 2, 1))
    assert np.array_equal(sf, s.transpose(0, 2, 1))


@pytest.mark.parametrize("L", [0, 1, 3, 6, 9])
def test_conv_state_window(oracle_mod, L):
    """Slab s of the window is the state after token L - W + s (zeros before the first
    token); only the last slab of the past window is read."""
    rng = np.random.default_rng(11)
    W, K = 4, 3
    x, w, bias, st = _case(rng, L=9, K=K)
    x = x[:, :L]
    past = rng.standard_normal((W,) + st.shape)
    y, win = oracle_mod.causal_conv(x, w, bias, past, silu=True, state_window=W)
    y0, s0 = oracle_mod.causal_conv(x, w, bias, past[W - 1], silu=True)
    assert np.array_equal(y, y0)
    if L == 0:
        assert np.array_equal(win, past)
        return
    assert np.array_equal(win[W - 1], s0)
    for s in range(W):
        token = L - W + s
        if token < 0:
            assert np.all(win[s] == 0.0)
        else:
            _, st_cut = oracle_mod.causal_conv(x[:, :token + 1], w, bias, past[W - 1])
            assert np.array_equal(win[s], st_cut)
    other = past.copy()
    other[:W - 1] = 123.0
    y2, win2 = oracle_mod.causal_conv(x, w, bias, other, silu=True, state_window=W)
    assert np.array_equal(y2, y) and np.array_equal(win2, win)


def test_conv_kernel_of_one_tap_is_pointwise(oracle_mod):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 5, 3))
    w = rng.standard_normal((3, 1, 1))
    bias = rng.standard_normal(3)
    y, s = oracle_mod.causal_conv(x, w, bias)
    assert _rel(y, x * w[:, 0, 0] + bias) < 1e-15
    assert s.shape == (2, 0, 3)


def test_conv_slots(oracle_mod):
    """Identity slots reproduce the plain call; unnamed pool entries stay bit-identical;
    relabelling the pool commutes; an out-of-range slot skips its row."""
    rng = np.random.default_rng(13)
    x, w, bias, st = _case(rng, B=3, L=4, K=4)
    y0, s0 = oracle_mod.causal_conv(x, w, bias, st, silu=True)
    y1, p1 = oracle_mod.conv_slots(x, w, st, [0, 1, 2], bias, silu=True)
    assert np.array_equal(y1, y0) and np.array_equal(p1, s0)
    pool = rng.standard_normal((6, 3, 5))
    slots = [4, 0, 2]
    y2, p2 = oracle_mod.conv_slots(x, w, pool, slots, bias, silu=True)
    for s in (1, 3, 5):
        assert np.array_equal(p2[s], pool[s])
    perm = rng.permutation(6)
    inv = np.argsort(perm)
    y3, p3 = oracle_mod.conv_slots(x, w, pool[perm], inv[slots], bias, silu=True)
    assert np.array_equal(y3, y2) and np.array_equal(p3, p2[perm])
    y4, p4 = oracle_mod.conv_slots(x, w, pool, [4, 6, 2], bias, silu=True)
    assert np.all(y4[1] == 0.0) and np.array_equal(p4[[0, 1, 3, 5]], pool[[0, 1, 3, 5]])


# ------------------------------------------------------------------ gated RMS norm

def test_norm_constant_row_closed_form(oracle_mod):
    """x = c everywhere: mean(x^2) = c^2, so y = c / sqrt(c^2 + eps) * scale * act(g)."""
    c, eps, width = -1.7, 0.3, 8
    rng = np.random.default_rng(20)
    scale = rng.standard_normal(width)
    g = rng.standard_normal((3, width))
    sig = 1.0 / (1.0 + np.exp(-g))
    for act, a in (("silu", g * sig), ("sigmoid", sig)):
        y = oracle_mod.gated_rmsnorm(np.full((3, width), c), scale, g, eps, act)
        assert _rel(y, c / np.sqrt(c * c + eps) * scale * a) < 1e-14


def test_norm_without_eps_is_scale_free_and_odd(oracle_mod):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((4, 16))
    scale = rng.standard_normal(16)
    g = rng.standard_normal((4, 16))
    y = oracle_mod.gated_rmsnorm(x, scale, g, 0.0)
    assert _rel(oracle_mod.gated_rmsnorm(7.5 * x, scale, g, 0.0), y) < 1e-14
    assert _rel(oracle_mod.gated_rmsnorm(-x, scale, g, 0.0), -y) < 1e-15


def test_norm_output_has_unit_rms_before_scale_and_gate(oracle_mod):
    """With eps = 0 and a gate far in sigmoid's saturation, y / scale has RMS 1."""
    rng = np.random.default_rng(22)
    x = rng.standard_normal((5, 32)) * 3.0
    scale = rng.uniform(0.5, 2.0, 32)
    y = oracle_mod.gated_rmsnorm(x, scale, np.full((5, 32), 60.0), 0.0, "sigmoid")
    assert np.max(np.abs(np.sqrt(np.mean((y / scale) ** 2, axis=1)) - 1.0)) < 1e-14


def test_norm_silu_is_sigmoid_times_gate(oracle_mod):
    rng = np.random.default_rng(23)
    x, g = rng.standard_normal((3, 12)), rng.standard_normal((3, 12))
    scale = rng.standard_normal(12)
    ys = oracle_mod.gated_rmsnorm(x, scale, g, 1e-5, "silu")
    yg = oracle_mod.gated_rmsnorm(x, scale, g, 1e-5, "sigmoid")
    assert _rel(ys, yg * g) < 1e-14


def test_norm_groups_are_consecutive_runs_of_the_scale_width(oracle_mod):
    """A last dimension of 3 groups normalises each run of `width` values on its own."""
    rng = np.random.default_rng(24)
    x, g = rng.standard_normal((2, 3 * 8)), rng.standard_normal((2, 3 * 8))
    scale = rng.standard_normal(8)
    y = oracle_mod.gated_rmsnorm(x, scale, g, 1e-5)
    for j in range(3):
        part = oracle_mod.gated_rmsnorm(x[:, 8 * j:8 * j + 8], scale, g[:, 8 * j:8 * j + 8], 1e-5)
        assert np.array_equal(y[:, 8 * j:8 * j + 8], part)
