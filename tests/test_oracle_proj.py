"""Pins of the projection oracle (no GPU): explicit sums on tiny inputs, identity weights that reduce the fused
projection to the step the other pins cover, and the row order of the stacked weight."""
import numpy as np

from oracle import attention as A
from oracle import proj as P

RNG = np.random.default_rng(99)


def test_projection_by_explicit_sums():
    """Each output is the sum over hidden units of x times the weight row, plus its bias: written as loops."""
    n, hidden, hq, hkv, d = 3, 5, 2, 1, 2
    x = RNG.standard_normal((n, hidden))
    w = RNG.standard_normal(((hq + 2 * hkv) * d, hidden))
    b = RNG.standard_normal((hq + 2 * hkv) * d)
    q, k, v = P.qkv_project(x, w, hq, hkv, d, b)
    flat = np.concatenate([q.reshape(n, -1), k.reshape(n, -1), v.reshape(n, -1)], axis=1)
    for t in range(n):
        for o in range(w.shape[0]):
            assert abs(flat[t, o] - (sum(x[t, i] * w[o, i] for i in range(hidden)) + b[o])) < 1e-12
    # rows of W: q heads first, then k, then v; head-major within each
    assert abs(k[1, 0, 1] - (x[1] @ w[hq * d + 1] + b[hq * d + 1])) < 1e-12
    assert abs(v[2, 0, 0] - (x[2] @ w[(hq + hkv) * d] + b[(hq + hkv) * d])) < 1e-12


def test_identity_weights_reduce_to_the_cache_update():
    """hidden = (Hq + 2 Hkv) d and W = I: the projected q, k, v are slices of x, so the fused step equals the
    cache update on those slices, bit for bit."""
    hq, hkv, d, n = 4, 2, 8, 5
    layer = A.Layer(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=d,
                    q_norm_w=1 + 0.1 * RNG.standard_normal(d), k_norm_w=1 + 0.1 * RNG.standard_normal(d))
    hidden = (hq + 2 * hkv) * d
    x = RNG.standard_normal((n, hidden))
    ang = RNG.uniform(-3, 3, (n, d // 2))
    cos, sin = np.cos(ang), np.sin(ang)
    rows, pos = [0, 1, 0, 1, 0], [0, 0, 1, 1, 2]
    kc1, vc1 = np.zeros((2, hkv, 4, d)), np.zeros((2, hkv, 4, d))
    kc2, vc2 = kc1.copy(), vc1.copy()
    got = P.project_and_update(layer, x, np.eye(hidden), rows, pos, cos, sin, kc1, vc1)
    want = A.kv_cache_update(layer, x[:, :hq * d].reshape(n, hq, d), x[:, hq * d:(hq + hkv) * d].reshape(n, hkv, d),
                             x[:, (hq + hkv) * d:].reshape(n, hkv, d), rows, pos, cos, sin, kc2, vc2)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(kc1, kc2)
    np.testing.assert_array_equal(vc1, vc2)


def test_o_projection():
    """o_proj concatenates the heads (head-major) and applies W_o^T plus the bias."""
    n, hq, d, hidden = 2, 3, 2, 4
    a = RNG.standard_normal((n, hq, d))
    w = RNG.standard_normal((hidden, hq * d))
    b = RNG.standard_normal(hidden)
    y = P.o_project(a, w, b)
    for t in range(n):
        for o in range(hidden):
            s = sum(a[t, h, j] * w[o, h * d + j] for h in range(hq) for j in range(d)) + b[o]
            assert abs(y[t, o] - s) < 1e-12
    np.testing.assert_array_equal(P.o_project(a, np.eye(hq * d)), a.reshape(n, -1))
