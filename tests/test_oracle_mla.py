"""Pins of the MLA oracle (no GPU): the absorbed form equals decompressing every head's keys and values
(the associativity the page "42. More models", "Serving it: absorbing the up-projections", rests on), the
deinterleaved split-half rotation equals rotating adjacent pairs, the page's per-token cache sizes, and the
YaRN temperature on the scale."""
import math

import numpy as np
from scipy.special import softmax as sp_softmax

from oracle import mla as M
from tests.conftest import read_golden

RNG = np.random.default_rng(2024)


def _angles(positions, r, theta=1e4):
    inv = theta ** (-np.arange(0, r, 2) / r)
    ang = np.outer(positions, inv)
    return np.cos(ang), np.sin(ang)


def test_absorbed_equals_decompressed():
    """Keys k_hj = [W_uk_h c_j, k_rope_j], values v_hj = W_uv_h c_j, ordinary softmax attention per head
    (brute force) against the absorbed form: W_uv_h applied to mla_decode's latent output."""
    H, nope, rope, vdim, rank, T = 4, 16, 8, 12, 20, 7
    c = RNG.standard_normal((T, rank))
    k_rope = RNG.standard_normal((T, rope))
    w_uk = RNG.standard_normal((H, nope, rank)) / math.sqrt(rank)
    w_uv = RNG.standard_normal((H, vdim, rank)) / math.sqrt(rank)
    q_nope = RNG.standard_normal((H, nope))
    q_rope = RNG.standard_normal((H, rope))
    pos = np.arange(T)
    p = T - 1
    cos, sin = _angles(pos, rope)
    kr = M.mla_rope(k_rope, cos, sin)                          # [T, rope]
    qr = M.mla_rope(q_rope[None], cos[p:p + 1], sin[p:p + 1])[0]
    scale = M.mla_scale(nope, rope)
    want = np.zeros((H, vdim))
    for h in range(H):
        z = [scale * (q_nope[h] @ (w_uk[h] @ c[j]) + qr[h] @ kr[j]) for j in range(T)]
        a = sp_softmax(np.array(z))
        want[h] = sum(a[j] * (w_uv[h] @ c[j]) for j in range(T))
    cache = np.zeros((1, T, rank + rope))
    M.mla_cache_update(c, k_rope, [0] * T, pos, cos, sin, cache)
    q_lat = np.einsum("hd,hdr->hr", q_nope, w_uk)
    q = M.mla_query(q_lat[None], q_rope[None], cos[p:p + 1], sin[p:p + 1])
    lat = M.mla_decode(q, cache, [0], [p], scale, rank)[0]     # [H, rank]
    got = np.einsum("hr,hvr->hv", lat, w_uv)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_deinterleaved_rotation_equals_adjacent_pair_rotation():
    """Rotating adjacent pairs (x_2i + i x_2i+1) by e^(i p w_i) and taking dot products gives what the
    deinterleaved split-half rotation gives: the cache may hold either order as long as q and k agree."""
    r = 8
    a, b = RNG.standard_normal((5, r)), RNG.standard_normal((5, r))
    pa, pb = np.array([3, 10, 0, 77, 5]), np.array([1, 4, 9, 2, 5])
    ca, sa = _angles(pa, r)
    cb, sb = _angles(pb, r)

    def adjacent(x, c, s):
        z = (x[:, 0::2] + 1j * x[:, 1::2]) * (c + 1j * s)
        out = np.empty_like(x)
        out[:, 0::2], out[:, 1::2] = z.real, z.imag
        return out

    want = np.einsum("nr,nr->n", adjacent(a, ca, sa), adjacent(b, cb, sb))
    got = np.einsum("nr,nr->n", M.mla_rope(a, ca, sa), M.mla_rope(b, cb, sb))
    np.testing.assert_allclose(got, want, atol=1e-12)
    np.testing.assert_array_equal(M.deinterleave(np.arange(8.0)), [0, 2, 4, 6, 1, 3, 5, 7])


def test_cache_sizes_golden():
    (ln,) = read_golden("mla_kv_bytes.txt")
    layers, heads, nope, rope, vdim, rank, full, mla_kib, saving = ln.split()
    layers, heads, nope, rope, vdim, rank = map(int, (layers, heads, nope, rope, vdim, rank))
    assert layers * heads * (nope + rope + vdim) * 2 == int(full)
    row = rank + rope                                          # one cached row per token and layer
    assert round(layers * row * 2 / 1024, 1) == float(mla_kib)
    assert round(int(full) / (layers * row * 2), 1) == float(saving)


def test_scale_and_yarn_temperature():
    """qk^-0.5 with qk = 128 + 64, times (0.1 * mscale_all_dim * ln s + 1)^2 under YaRN (DeepSeek-V3: s = 40)."""
    assert M.mla_scale(128, 64) == 192 ** -0.5
    sc = {"type": "yarn", "factor": 40, "mscale": 1.0, "mscale_all_dim": 1.0}
    np.testing.assert_allclose(M.mla_scale(128, 64, sc), 192 ** -0.5 * (0.1 * math.log(40) + 1) ** 2, rtol=1e-15)
    assert M.mla_scale(128, 64, {"factor": 1.0, "mscale_all_dim": 1.0}) == 192 ** -0.5


def test_one_visible_row_and_window_one():
    """A query that sees one row gets that row's latent, whatever its scores."""
    rank, rope = 6, 4
    cache = RNG.standard_normal((2, 5, rank + rope))
    q = RNG.standard_normal((2, 3, rank + rope)) * 10
    out = M.mla_decode(q, cache, [1, 0], [0, 4], 0.3, rank, window=0)
    np.testing.assert_allclose(out[0], np.broadcast_to(cache[1, 0, :rank], (3, rank)), atol=1e-15)
    out = M.mla_decode(q, cache, [1, 0], [3, 4], 0.3, rank, window=1)
    np.testing.assert_allclose(out[1], np.broadcast_to(cache[0, 4, :rank], (3, rank)), atol=1e-15)
