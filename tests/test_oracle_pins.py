"""Pins of the fp64 oracle against what the pages and the mathematics fix (no GPU).

Each test names the fact it checks and where it comes from. They are chosen so that a plausible slip in
the oracle (a wrong exponent, swapped blend weights, a dropped factor, a transposed head mapping, an
off-by-one window) fails at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from oracle import attention as O
from tests.conftest import read_golden

RNG = np.random.default_rng(12345)


# ------------------------------------------------------------------ frequencies

def test_slowest_wavelength_and_pair0():
    """Page 1 "Scaled RoPE": theta 500000, d 128 -> slowest pair wavelength about 2.6 M positions;
    pair 0 turns once every 2*pi positions."""
    theta, d, wl_last, wl0 = read_golden("rope_slowest_wavelength.txt")[0].split()
    inv, af = O.rope_inv_freq(int(d), float(theta))
    assert af == 1.0 and inv.shape == (int(d) // 2,)
    wl = 2 * math.pi / inv
    assert round(wl[-1] / 1e5) * 1e5 == float(wl_last)
    assert wl[0] == pytest.approx(float(wl0), rel=1e-15)
    assert np.all(np.diff(inv) < 0)          # pairs slow down monotonically


def test_llama3_pair_split():
    """Page 1 "Scaled RoPE", Llama 3 bullet: kept / blended / divided pair ranges, derived by hand."""
    k0, k1, b0, b1, d0, d1 = map(int, read_golden("llama3_pair_split.txt")[0].split())
    sc = {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
          "original_max_position_embeddings": 8192}
    base, _ = O.rope_inv_freq(128, 5e5)
    inv, af = O.rope_inv_freq(128, 5e5, sc)
    assert af == 1.0
    ratio = inv / base
    np.testing.assert_array_equal(ratio[k0:k1 + 1], 1.0)
    np.testing.assert_allclose(ratio[d0:d1 + 1], 1 / 8.0, rtol=1e-15)
    mid = ratio[b0:b1 + 1]
    assert np.all((mid > 1 / 8.0) & (mid < 1.0))
    # the blend moves from "kept" to "divided" as the wavelength grows (no jump, no reversal)
    assert np.all(np.diff(ratio) <= 0)


@pytest.mark.parametrize("kind", ["linear", "llama3"])
def test_factor_one_is_unscaled(kind):
    """North star: rope_scaling factor 1 equals unscaled RoPE."""
    sc = {"rope_type": kind, "factor": 1.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
          "original_max_position_embeddings": 8192}
    base, _ = O.rope_inv_freq(128, 5e5)
    inv, af = O.rope_inv_freq(128, 5e5, sc)
    np.testing.assert_allclose(inv, base, rtol=4e-16, atol=0)     # equal up to the blend's rounding
    assert af == 1.0


def test_linear_is_position_interpolation():
    """Page 1 "Scaled RoPE": linear scaling makes position p look like p / s."""
    s = 4.0
    inv_l, _ = O.rope_inv_freq(64, 1e4, {"type": "linear", "factor": s})
    inv_d, _ = O.rope_inv_freq(64, 1e4)
    p = np.array([0, 3, 17, 1000, 4095])
    cl, sl = O.rope_tables(p, inv_l, 1.0)
    cd, sd = O.rope_tables(p / s, inv_d, 1.0)
    np.testing.assert_allclose(cl, cd, atol=1e-13)
    np.testing.assert_allclose(sl, sd, atol=1e-13)


def test_longrope_switch_and_divisors():
    """"Model resolution": short factors while the sequence is within original_max_position_embeddings,
    long ones past it (reading R2: per-pair divisors, chosen by the sequence length)."""
    r = O.rotary_dim(128, 0.75)
    assert r == 96                                   # workload 5: 48 factors per list = r/2
    short = np.linspace(1.0, 1.2, r // 2)
    long_ = np.linspace(1.0, 40.0, r // 2)
    sc = {"rope_type": "longrope", "short_factor": short, "long_factor": long_,
          "original_max_position_embeddings": 4096}
    base, _ = O.rope_inv_freq(r, 1e4)
    inv_s, af_s = O.rope_inv_freq(r, 1e4, sc, 131072, seq_len=4096)
    inv_l, af_l = O.rope_inv_freq(r, 1e4, sc, 131072, seq_len=4097)
    np.testing.assert_allclose(inv_s, base / short, rtol=1e-15)
    np.testing.assert_allclose(inv_l, base / long_, rtol=1e-15)
    # attention factor sqrt(1 + ln 32 / ln 4096) = sqrt(1 + 5/12) in closed form (reading R11)
    assert af_s == af_l == pytest.approx(math.sqrt(17.0 / 12.0), rel=1e-15)
    # all-ones tables and factor 1 reduce to the default table
    ones = {"rope_type": "longrope", "short_factor": np.ones(r // 2), "long_factor": np.ones(r // 2),
            "original_max_position_embeddings": 4096, "attention_factor": 1.0}
    inv1, af1 = O.rope_inv_freq(r, 1e4, ones, 131072, seq_len=10000)
    np.testing.assert_array_equal(inv1, base)
    assert af1 == 1.0
    # a uniform divisor table equals linear scaling by that factor
    two = {"rope_type": "longrope", "short_factor": np.full(r // 2, 2.0), "long_factor": np.full(r // 2, 2.0),
           "original_max_position_embeddings": 4096, "attention_factor": 1.0}
    inv2, _ = O.rope_inv_freq(r, 1e4, two, 131072, seq_len=10)
    lin, _ = O.rope_inv_freq(r, 1e4, {"type": "linear", "factor": 2.0})
    np.testing.assert_allclose(inv2, lin, rtol=1e-15)
    # no extension (max = original): factor 1
    _, af0 = O.rope_inv_freq(r, 1e4, sc, 4096, seq_len=10)
    assert af0 == 1.0


def test_yarn_ramp_and_temperature():
    """Page 1 "Scaled RoPE", YaRN bullet: pairs that turn more than beta_fast (32) times over the original
    context are kept, pairs that turn fewer than beta_slow (1) times are interpolated, a ramp between;
    cos and sin are multiplied by 0.1 ln s + 1."""
    old, s = 4096, 8.0
    sc = {"rope_type": "yarn", "factor": s, "original_max_position_embeddings": old}
    base, _ = O.rope_inv_freq(128, 1e4)
    inv, af = O.rope_inv_freq(128, 1e4, sc, 32768)
    assert af == pytest.approx(0.1 * math.log(s) + 1.0, rel=1e-15)
    turns = old * base / (2 * math.pi)
    np.testing.assert_array_equal(inv[turns >= 32], base[turns >= 32])
    np.testing.assert_allclose(inv[turns <= 1], base[turns <= 1] / s, rtol=1e-15)
    ratio = inv / base
    assert np.all(np.diff(ratio) <= 1e-15)
    # factor defaults to max_position_embeddings / original
    inv_d, _ = O.rope_inv_freq(128, 1e4, {"rope_type": "yarn", "original_max_position_embeddings": old}, 32768)
    np.testing.assert_array_equal(inv_d, inv)


def _yarn_golden():
    return {k: float(v) for k, v in (ln.split() for ln in read_golden("yarn_ramp.txt"))}


@pytest.mark.parametrize("truncate", [True, False])
def test_yarn_ramp_golden(truncate):
    """Page 1 "Scaled RoPE", yarn branch of rope_inv_freq, values derived by hand in the fixture: the
    fractional pair index of 32 and 1 rotations over the original context, floor/ceil of the two ends
    unless truncate is false, a ramp linear in the pair index between them."""
    g = _yarn_golden()
    tag = "truncate" if truncate else "no_truncate"
    sc = {"rope_type": "yarn", "factor": 32.0, "original_max_position_embeddings": 4096,
          "beta_fast": 32, "beta_slow": 1, "truncate": truncate}
    base, _ = O.rope_inv_freq(128, 1e4)
    inv, _ = O.rope_inv_freq(128, 1e4, sc)
    ratio = inv / base
    for i in (25, 33, 40):
        assert ratio[i] == pytest.approx(g[f"ratio_{tag}_{i}"], abs=2e-9)
    lo, hi = g[f"lo_{tag}"], g[f"hi_{tag}"]
    i = np.arange(64)
    np.testing.assert_allclose(ratio[i <= lo], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(ratio[i >= hi], g["ratio_slow_end"], rtol=1e-15)
    # the ramp is linear in i: recover its two ends from the interior and compare with the fixture
    ramp = (1.0 - ratio) * 32.0 / 31.0
    inner = (i > lo) & (i < hi)
    slope, icpt = np.polyfit(i[inner], ramp[inner], 1)
    np.testing.assert_allclose(ramp[inner], slope * i[inner] + icpt, atol=1e-12)
    assert -icpt / slope == pytest.approx(lo, abs=1e-8)
    assert (1.0 - icpt) / slope == pytest.approx(hi, abs=1e-8)
    if not truncate:
        assert lo == pytest.approx(g["dim_for_beta_fast"], abs=1e-9)
        assert hi == pytest.approx(g["dim_for_beta_slow"], abs=1e-9)


def test_yarn_attention_factor_golden():
    """Page 1 "Scaled RoPE", yarn branch: the attention factor is mscale(s, mscale) / mscale(s, mscale_all_dim)
    when both are stated, else mscale(s) = 0.1 ln s + 1; a stated attention_factor wins."""
    g = _yarn_golden()
    sc = {"rope_type": "yarn", "factor": 32.0, "original_max_position_embeddings": 4096}
    _, af_pair = O.rope_inv_freq(128, 1e4, dict(sc, mscale=0.707, mscale_all_dim=1.0605))
    _, af_alone = O.rope_inv_freq(128, 1e4, dict(sc, mscale=0.707))
    _, af_none = O.rope_inv_freq(128, 1e4, sc)
    _, af_given = O.rope_inv_freq(128, 1e4, dict(sc, mscale=0.707, mscale_all_dim=1.0605, attention_factor=1.25))
    assert af_pair == pytest.approx(g["attention_mscale_pair"], abs=2e-9)
    assert af_alone == pytest.approx(g["attention_mscale_alone"], abs=2e-9)
    assert af_none == pytest.approx(g["attention_mscale_alone"], abs=2e-9)
    assert af_given == 1.25


def test_unknown_kind_refused():
    """Page 1 rope_inv_freq: an unimplemented type raises ValueError naming it."""
    with pytest.raises(ValueError, match="dynamic"):
        O.rope_inv_freq(64, 1e4, {"type": "dynamic", "factor": 2.0})


# ------------------------------------------------------------------ rotation

def _rand(*shape):
    return RNG.standard_normal(shape)


def test_rope_pairing_and_pair0_angle():
    """Page 3 §4: a 64-wide head is split into 32 pairs, feature i with feature i + 32, pair i rotated by
    m * theta_i; page 1: pair 0 turns once every 2 pi positions (theta_0 = 1)."""
    inv, af = O.rope_inv_freq(64, 1e4)
    for m in (1, 2, 7, 100):
        c, s = O.rope_tables([m], inv, af)
        e0 = np.zeros(64)
        e0[0] = 1.0
        y = O.apply_rope(e0[None], c, s)[0]
        assert y[0] == pytest.approx(math.cos(m), abs=1e-15)
        assert y[32] == pytest.approx(math.sin(m), abs=1e-15)
        assert np.count_nonzero(np.abs(y) > 1e-15) <= 2      # only its partner is touched
        e32 = np.zeros(64)
        e32[32] = 1.0
        y = O.apply_rope(e32[None], c, s)[0]
        assert y[0] == pytest.approx(-math.sin(m), abs=1e-15)
        assert y[32] == pytest.approx(math.cos(m), abs=1e-15)


def test_rope_is_complex_multiplication():
    """Split-half rotation equals multiplying (x_i + i x_{i+r/2}) by exp(i p inv_i)."""
    r, d = 96, 128
    inv, _ = O.rope_inv_freq(r, 1e4)
    p = np.array([0, 1, 4095, 4097, 65535])
    c, s = O.rope_tables(p, inv, 1.0)
    x = _rand(len(p), d)
    y = O.apply_rope(x, c, s)
    z = (x[:, :r // 2] + 1j * x[:, r // 2:r]) * np.exp(1j * p[:, None] * inv[None, :])
    np.testing.assert_allclose(y[:, :r // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[:, r // 2:r], z.imag, atol=1e-12)
    np.testing.assert_array_equal(y[:, r:], x[:, r:])      # pass-through dims untouched (R3)


def test_rope_norm_and_identity_and_factor():
    """Rotation preserves each pair's norm (times af^2); position 0 is the identity times af on the rotated
    dims; the attention factor leaves pass-through dims alone (R3)."""
    r, d, af = 96, 128, 1.190238
    inv, _ = O.rope_inv_freq(r, 1e4)
    x = _rand(6, d)
    p = np.array([0, 5, 99, 4096, 70000, 131071])
    c, s = O.rope_tables(p, inv, af)
    y = O.apply_rope(x, c, s)
    h = r // 2
    n_in = x[:, :h] ** 2 + x[:, h:r] ** 2
    n_out = y[:, :h] ** 2 + y[:, h:r] ** 2
    np.testing.assert_allclose(n_out, af * af * n_in, rtol=1e-12)
    np.testing.assert_allclose(y[0, :r], af * x[0, :r], rtol=1e-15)
    np.testing.assert_array_equal(y[:, r:], x[:, r:])


def test_rope_relative_position():
    """North star: unscaled q.k after RoPE depends only on the position difference."""
    d = 128
    inv, af = O.rope_inv_freq(d, 5e5)
    q, k = _rand(d), _rand(d)
    for p, pk, delta in [(10, 3, 1000), (5000, 4999, 77777), (0, 0, 123)]:
        c, s = O.rope_tables([p, pk, p + delta, pk + delta], inv, af)
        qa = O.apply_rope(q[None], c[0:1], s[0:1])[0]
        ka = O.apply_rope(k[None], c[1:2], s[1:2])[0]
        qb = O.apply_rope(q[None], c[2:3], s[2:3])[0]
        kb = O.apply_rope(k[None], c[3:4], s[3:4])[0]
        assert qa @ ka == pytest.approx(qb @ kb, abs=1e-10)


# ------------------------------------------------------------------ norm

def test_rmsnorm_closed_forms():
    """Page 3 §3.2: each vector is rescaled to RMS 1, then times the gain."""
    x = _rand(5, 3, 128)
    y = O.rms_norm(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, np.ones(128), 0.0), y, rtol=1e-13)   # scale free
    c, eps = 0.3, 1e-6
    w = 1.0 + 0.02 * _rand(128)
    y = O.rms_norm(np.full(128, c), w, eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps) * w, rtol=1e-15)


# ------------------------------------------------------------------ mask and attention

def _golden_masks():
    lines = read_golden("window_masks.txt")
    out, w, rows = {}, None, []
    for ln in lines:
        if ln.startswith("w="):
            if w is not None:
                out[w] = np.array(rows, dtype=bool)
            w, rows = int(ln[2:]), []
        else:
            rows.append([ch == "1" for ch in ln])
    out[w] = np.array(rows, dtype=bool)
    return out


def test_window_masks_golden():
    """Page 1 "Sliding windows": keys more than w - 1 positions back are masked (R8)."""
    pos = np.arange(6)
    for w, mask in _golden_masks().items():
        np.testing.assert_array_equal(O.window_allowed(pos, pos, w), mask)
    np.testing.assert_array_equal(O.window_allowed(pos, pos, 6), _golden_masks()[0])   # w >= T is full
    np.testing.assert_array_equal(O.window_allowed([3], [-1, 2, -1, 3], 0), [[False, True, False, True]])


def _bruteforce(q, k, v, masks, scale, cap=0.0, sinks=None):
    """Per query and head: softmax over the explicitly listed visible keys (scipy's softmax); with sinks, the
    head's sink logit joins the list and its weight is then dropped."""
    T, hq, d = q.shape
    hkv = k.shape[0]
    out = np.zeros_like(q)
    for t in range(T):
        for h in range(hq):
            g = h * hkv // hq
            js = [j for j in range(k.shape[1]) if masks[t, j]]
            if not js:
                continue
            z = np.array([scale * float(np.dot(q[t, h], k[g, j])) for j in js])
            if cap:
                z = cap * np.tanh(z / cap)
            w = sp_softmax(z) if sinks is None else sp_softmax(np.append(z, sinks[h]))[:-1]
            out[t, h] = sum(wi * v[g, j] for wi, j in zip(w, js))
    return out


@pytest.mark.parametrize("w", [0, 1, 2, 3])
def test_attention_bruteforce_tiny(w):
    """Brute force on tiny inputs with the hand-written masks: T = 6, Hq = 4, Hkv = 2 (GQA), d = 8."""
    T, hq, hkv, d = 6, 4, 2, 8
    q, k, v = _rand(T, hq, d), _rand(hkv, T, d), _rand(hkv, T, d)
    pos = np.arange(T)
    masks = _golden_masks()[w]
    got = O.causal_attention(q, k, v, pos, pos, window=w)
    np.testing.assert_allclose(got, _bruteforce(q, k, v, masks, 1 / math.sqrt(d)), atol=1e-13)
    got = O.causal_attention(q, k, v, pos, pos, window=w, softcap=0.7)
    np.testing.assert_allclose(got, _bruteforce(q, k, v, masks, 1 / math.sqrt(d), cap=0.7), atol=1e-13)


# ------------------------------------------------------------------ learned sinks (page "Model resolution", gpt_oss)

def test_sink_single_key_is_a_sigmoid():
    """One visible key and a sink: the key's weight is e^z / (e^z + e^s) = 1 / (1 + e^(s - z)); the rest of the
    mass (the sink's share) reaches no value."""
    d = 16
    q, k, v = _rand(1, 3, d), _rand(3, 1, d), _rand(3, 1, d)
    sinks = np.array([-1.5, 0.25, 3.0])
    got = O.causal_attention(q, k, v, [0], [0], sinks=sinks)
    for h in range(3):
        z = float(np.dot(q[0, h], k[h, 0])) / math.sqrt(d)
        np.testing.assert_allclose(got[0, h], v[h, 0] / (1.0 + math.exp(sinks[h] - z)), atol=1e-15)


@pytest.mark.parametrize("w,cap", [(0, 0.0), (2, 0.0), (0, 0.7), (3, 0.7)])
def test_sink_bruteforce_tiny(w, cap):
    """Brute force with the sink as one more softmax entry whose weight is dropped: GQA, windows, and a
    soft-cap that applies to the scores but not to the sink (sinks up to 2.5 lie beyond a 0.7 cap)."""
    T, hq, hkv, d = 6, 4, 2, 8
    q, k, v = _rand(T, hq, d), _rand(hkv, T, d), _rand(hkv, T, d)
    pos = np.arange(T)
    sinks = np.array([0.3, -2.0, 2.5, 1.1])
    got = O.causal_attention(q, k, v, pos, pos, window=w, softcap=cap, sinks=sinks)
    want = _bruteforce(q, k, v, _golden_masks()[w], 1 / math.sqrt(d), cap=cap, sinks=sinks)
    np.testing.assert_allclose(got, want, atol=1e-13)


def test_sink_at_minus_infinity_is_no_sink():
    """A sink of -inf has weight 0: the result is the plain softmax, bit for bit."""
    q, k, v = _rand(5, 4, 16), _rand(2, 5, 16), _rand(2, 5, 16)
    pos = np.arange(5)
    np.testing.assert_array_equal(O.causal_attention(q, k, v, pos, pos, window=3, sinks=np.full(4, -np.inf)),
                                  O.causal_attention(q, k, v, pos, pos, window=3))


def test_sink_share_with_unit_values():
    """With every value equal to 1 the output is the mass the keys keep: 1 - 1 / (1 + sum_j e^(z_j - s))."""
    T, d = 4, 8
    q, k = _rand(T, 2, d), _rand(1, T, d)
    v = np.ones((1, T, d))
    pos = np.arange(T)
    sinks = np.array([0.5, -0.75])
    got = O.causal_attention(q, k, v, pos, pos, sinks=sinks)
    for t in range(T):
        for h in range(2):
            zs = [float(np.dot(q[t, h], k[0, j])) / math.sqrt(d) for j in range(t + 1)]
            keep = 1.0 - 1.0 / (1.0 + sum(math.exp(z - sinks[h]) for z in zs))
            np.testing.assert_allclose(got[t, h], np.full(d, keep), atol=1e-14)


def test_default_scale_is_inverse_sqrt_d():
    """Page 3 §3.4: logits are divided by sqrt(d_h) (by 8 for d_h = 64)."""
    q, k, v = _rand(5, 2, 64), _rand(2, 5, 64), _rand(2, 5, 64)
    pos = np.arange(5)
    np.testing.assert_array_equal(O.causal_attention(q, k, v, pos, pos),
                                  O.causal_attention(q, k, v, pos, pos, scale=1 / 8.0))


def test_equal_keys_give_mean_of_values():
    """Equal logits give uniform weights: the output is the mean of the visible values."""
    T, d = 7, 16
    q = _rand(T, 2, d)
    k = np.repeat(_rand(1, 1, d), T, axis=1)
    v = _rand(1, T, d)
    pos = np.arange(T)
    for w in (0, 3):
        got = O.causal_attention(q, k, v, pos, pos, window=w)
        for t in range(T):
            lo = max(0, t - w + 1) if w else 0
            np.testing.assert_allclose(got[t, 0], v[0, lo:t + 1].mean(axis=0), atol=1e-14)


def test_window_one_is_own_value():
    """w = 1: each query sees only its own key, so its output is its own value."""
    q, k, v = _rand(9, 4, 32), _rand(1, 9, 32), _rand(1, 9, 32)
    pos = np.arange(9)
    got = O.causal_attention(q, k, v, pos, pos, window=1)
    np.testing.assert_allclose(got, np.broadcast_to(v[0][:, None, :], got.shape), atol=1e-15)


def test_softcap_limits():
    """Soft-cap (R5): cap -> infinity is uncapped; a key with an unbounded logit against one with logit 0
    gets weight sigmoid(cap) exactly in the limit (the capped logits are cap and 0)."""
    q, k, v = _rand(6, 2, 32), _rand(2, 6, 32), _rand(2, 6, 32)
    pos = np.arange(6)
    np.testing.assert_allclose(O.causal_attention(q, k, v, pos, pos, softcap=1e9),
                               O.causal_attention(q, k, v, pos, pos), atol=1e-12)
    cap = 1.3
    qq = np.zeros((1, 1, 4))
    qq[0, 0, 0] = 1.0
    kk = np.zeros((1, 2, 4))
    kk[0, 0, 0] = 1e12                      # logit 5e11 before the cap
    vv = np.array([[[1.0, 0, 0, 0], [0, 1.0, 0, 0]]])
    o = O.causal_attention(qq, kk, vv, [1], [0, 1], softcap=cap)
    sig = 1.0 / (1.0 + math.exp(-cap))
    np.testing.assert_allclose(o[0, 0, :2], [sig, 1 - sig], rtol=1e-14)


def test_gqa_equals_mha_with_repeated_heads():
    """GQA (R4): query head h reads KV head floor(h / G); the same as MHA over KV heads repeated G times
    each (contiguous groups)."""
    T, hq, hkv, d = 10, 6, 2, 16
    q, k, v = _rand(T, hq, d), _rand(hkv, T, d), _rand(hkv, T, d)
    pos = np.arange(T)
    got = O.causal_attention(q, k, v, pos, pos, window=4)
    rep = O.causal_attention(q, np.repeat(k, hq // hkv, axis=0), np.repeat(v, hq // hkv, axis=0), pos, pos, window=4)
    np.testing.assert_allclose(got, rep, atol=1e-15)
    wrong = O.causal_attention(q, np.tile(k, (hq // hkv, 1, 1)), np.tile(v, (hq // hkv, 1, 1)), pos, pos, window=4)
    assert np.max(np.abs(got - wrong)) > 1e-3            # the other mapping is distinguishable


def test_no_visible_key_gives_zero():
    """R7: a query with no visible key returns 0 (never NaN)."""
    q, k, v = _rand(2, 2, 8), _rand(1, 3, 8), _rand(1, 3, 8)
    o = O.causal_attention(q, k, v, [5, 6], [-1, -1, -1])
    np.testing.assert_array_equal(o, 0.0)


# ------------------------------------------------------------------ the step: cache, prefill, decode

def _layer(d=32, hq=4, hkv=2, r=None, window=0, softcap=0.0, norm=False):
    r = r or d
    return O.Layer(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=r,
                   q_norm_w=(1 + 0.02 * _rand(d)) if norm else None,
                   k_norm_w=(1 + 0.02 * _rand(d)) if norm else None, window=window, softcap=softcap)


def _rope(layer, pos, L):
    spec = O.RopeSpec(theta=1e4)
    return O.rope_tables_for_tokens(spec, layer.rotary_dim, pos, L)


def test_cache_update_writes_only_its_slots():
    """Page 3 §3.3 / page 1 cache.update: k_rot and v land at (row, position); v is stored unchanged;
    every other slot keeps its sentinel."""
    L = _layer(norm=True, r=24)
    R, M, n = 3, 16, 5
    kc = np.full((R, 2, M, 32), 7.25)
    vc = np.full((R, 2, M, 32), -3.5)
    q, k, v = _rand(n, 4, 32), _rand(n, 2, 32), _rand(n, 2, 32)
    rows = np.array([2, 0, 2, 1, 0])
    pos = np.array([4, 0, 5, 15, 1])
    c, s = _rope(L, pos, pos + 1)
    q_rot = O.kv_cache_update(L, q, k, v, rows, pos, c, s, kc, vc)
    for t in range(n):
        np.testing.assert_array_equal(vc[rows[t], :, pos[t]], v[t])
        kn = O.rms_norm(k[t], L.k_norm_w, L.eps)
        np.testing.assert_allclose(kc[rows[t], :, pos[t]], O.apply_rope(kn, c[t:t + 1], s[t:t + 1]), atol=1e-14)
        qn = O.rms_norm(q[t], L.q_norm_w, L.eps)
        np.testing.assert_allclose(q_rot[t], O.apply_rope(qn, c[t:t + 1], s[t:t + 1]), atol=1e-14)
    written = np.zeros((R, M), dtype=bool)
    written[rows, pos] = True
    assert np.all(kc.transpose(0, 2, 1, 3)[~written] == 7.25)
    assert np.all(vc.transpose(0, 2, 1, 3)[~written] == -3.5)


@pytest.mark.parametrize("window,cap", [(0, 0.0), (5, 0.0), (0, 2.0), (3, 1.5)])
def test_decode_equals_prefill_row(window, cap):
    """Page 3 (tests/test_sanity.py list): cached decoding equals recomputing the whole sequence. Token t
    decoded against the cache equals row t of a one-shot prefill of tokens 0..t."""
    L = _layer(window=window, softcap=cap, norm=True, r=16)
    T, M = 12, 12
    q, k, v = _rand(T, 4, 32), _rand(T, 2, 32), _rand(T, 2, 32)
    pos = np.arange(T)
    c, s = _rope(L, pos, np.full(T, T))
    kc, vc = np.zeros((1, 2, M, 32)), np.zeros((1, 2, M, 32))
    q_rot = O.kv_cache_update(L, q, k, v, np.zeros(T, int), pos, c, s, kc, vc)
    full = O.attn_prefill(L, q_rot, kc, vc, [0, T], [0], [0])
    # decode: tokens one at a time into a fresh cache
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    for t in range(T):
        qr = O.kv_cache_update(L, q[t:t + 1], k[t:t + 1], v[t:t + 1], [0], [t], c[t:t + 1], s[t:t + 1], kc2, vc2)
        o = O.attn_decode(L, qr, kc2, vc2, [0], [t])
        np.testing.assert_allclose(o[0], full[t], atol=1e-13)
        o1 = O.attn_decode_one(L, qr[0], kc2[0], vc2[0], t)
        np.testing.assert_allclose(o1, full[t], atol=1e-13)


def test_chunked_prefill_equals_one_shot():
    """Chunks at first_pos see the earlier chunks' keys in the cache: chunked == one-shot."""
    L = _layer(window=4, norm=False)
    T = 11
    q, k, v = _rand(T, 4, 32), _rand(T, 2, 32), _rand(T, 2, 32)
    pos = np.arange(T)
    c, s = _rope(L, pos, np.full(T, T))
    kc, vc = np.zeros((2, 2, T, 32)), np.zeros((2, 2, T, 32))
    q_rot = O.kv_cache_update(L, q, k, v, np.ones(T, int), pos, c, s, kc, vc)
    full = O.attn_prefill(L, q_rot, kc, vc, [0, T], [1], [0])
    parts = []
    for a, b in [(0, 3), (3, 4), (4, 11)]:
        parts.append(O.attn_prefill(L, q_rot[a:b], kc, vc, [0, b - a], [1], [a]))
    np.testing.assert_allclose(np.concatenate(parts), full, atol=1e-14)
    # two sequences in one call, in different rows, equal two separate calls
    kc[0] = kc[1]
    vc[0] = vc[1]
    both = O.attn_prefill(L, np.concatenate([q_rot[:4], q_rot[:7]]), kc, vc, [0, 4, 11], [0, 1], [0, 0])
    np.testing.assert_allclose(both[:4], full[:4], atol=1e-14)
    np.testing.assert_allclose(both[4:], full[:7], atol=1e-14)


def test_key_positions_decide_not_slots():
    """Page 1 DecoderAttention.forward: with key_positions the mask compares positions, so a row whose
    slots are permuted (positions permuted alike) gives the same output; -1 marks an empty slot."""
    L = _layer(window=5)
    T = 9
    q_rot, kk, vv = _rand(T, 4, 32), _rand(1, 2, T, 32), _rand(1, 2, T, 32)
    base = O.attn_prefill(L, q_rot, kk, vv, [0, T], [0], [0])
    perm = RNG.permutation(T)
    kp = np.full((1, T + 3), -1)
    kp[0, :T] = perm
    kk2 = np.zeros((1, 2, T + 3, 32))
    vv2 = np.zeros((1, 2, T + 3, 32))
    kk2[0, :, :T] = kk[0][:, perm]
    vv2[0, :, :T] = vv[0][:, perm]
    kk2[0, :, T:] = 1e30                      # empty slots must not be read into the result
    got = O.attn_prefill(L, q_rot, kk2, vv2, [0, T], [0], [0], key_positions=kp)
    np.testing.assert_allclose(got, base, atol=1e-14)


def test_kv_bytes_per_token_golden():
    """Page 1 "Multi-head latent attention": KV KiB per token of real configurations; the step stores one
    bf16 K and V vector of head_dim per KV head per layer."""
    for ln in read_golden("kv_bytes_per_token.txt"):
        model, layers, hkv, d, kib = ln.split()
        per_key_layer = 2 * int(hkv) * int(d) * 2          # K and V, bf16
        assert int(layers) * per_key_layer / 1024 == float(kib), model
