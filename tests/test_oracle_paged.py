"""Pins of the oracle's paged KV cache (no GPU): the slot mapping written out by hand, the special case of
one block per (row, block index) in order that reduces to the contiguous cache, invariance under any
placement of the blocks, and recycling of blocks that lie wholly before every query's window."""
import math

import numpy as np
import pytest

from oracle import attention as O
from tests.conftest import read_golden

RNG = np.random.default_rng(777)


def _rand(*shape):
    return RNG.standard_normal(shape)


def test_slot_mapping_golden():
    """Each slot of the pool holds a distinct number; paged_view returns the ones the hand-written list names."""
    bs, hkv, d = 4, 1, 1
    pool = np.arange(5 * hkv * bs * d, dtype=float).reshape(5, hkv, bs, d)
    table = np.array([[2, 0, -1], [1, 3, 4]])
    for ln in read_golden("paged_slots.txt"):
        row, pos, blk, off = map(int, ln.split())
        got = O.paged_view(pool, table, bs, row, pos, pos + 1)[0, 0, 0]
        assert got == pool[blk, 0, off, 0], (row, pos)
    with pytest.raises(ValueError):
        O.paged_view(pool, table, bs, 0, 8, 9)          # block index 2 of row 0 is unmapped


def _contiguous_to_paged(kc, bs, rng):
    """Split a contiguous cache [R, Hkv, M, d] into blocks placed in random order in a pool with spare blocks."""
    R, hkv, M, d = kc.shape
    nb = math.ceil(M / bs)
    n_blocks = R * nb + 3
    perm = rng.permutation(n_blocks)[:R * nb].reshape(R, nb)
    pool = np.full((n_blocks, hkv, bs, d), np.nan)
    for r in range(R):
        for b in range(nb):
            seg = kc[r, :, b * bs:(b + 1) * bs]
            pool[perm[r, b], :, :seg.shape[1]] = seg
    return pool, perm


def _layer(hq, hkv, d, window=0, softcap=0.0, sinks=None):
    return O.Layer(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=d, window=window,
                   softcap=softcap, sinks=sinks)


@pytest.mark.parametrize("window,bs", [(0, 4), (5, 4), (3, 8)])
def test_paged_equals_contiguous(window, bs):
    """A paged pool holding the contiguous cache's blocks (in any order) gives the contiguous results."""
    R, hq, hkv, d, M = 3, 4, 2, 8, 21
    kc, vc = _rand(R, hkv, M, d), _rand(R, hkv, M, d)
    rng = np.random.default_rng(5)
    kp, perm = _contiguous_to_paged(kc, bs, rng)
    vp = np.full_like(kp, np.nan)
    for r in range(R):
        for b in range(perm.shape[1]):
            seg = vc[r, :, b * bs:(b + 1) * bs]
            vp[perm[r, b], :, :seg.shape[1]] = seg
    layer = _layer(hq, hkv, d, window=window, sinks=np.array([0.1, -0.5, 1.0, -3.0]))
    lens = [7, 1, 5]
    first = [14, 0, 9]
    q_start = np.concatenate([[0], np.cumsum(lens)])
    q = _rand(int(q_start[-1]), hq, d)
    rows = [2, 0, 1]
    want = O.attn_prefill(layer, q, kc, vc, q_start, rows, first)
    got = O.attn_prefill_paged(layer, q, kp, vp, perm, bs, q_start, rows, first)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)     # a window sums fewer masked zeros
    pos = [20, 0, 13]
    qd = _rand(3, hq, d)
    np.testing.assert_allclose(O.attn_decode_paged(layer, qd, kp, vp, perm, bs, rows, pos),
                               O.attn_decode(layer, qd, kc, vc, rows, pos), rtol=0, atol=1e-13)


def test_out_of_window_blocks_may_be_recycled():
    """With a window w, a block wholly before p - w + 1 for every query of a call is never read: unmapping it
    (its slot in the table = -1, the block's contents garbage) leaves the results as they were."""
    R, hq, hkv, d, M, bs, w = 2, 2, 1, 8, 40, 4, 6
    kc, vc = _rand(R, hkv, M, d), _rand(R, hkv, M, d)
    table = np.arange(R * (M // bs)).reshape(R, M // bs)
    kp = kc.reshape(R, hkv, M // bs, bs, d).transpose(0, 2, 1, 3, 4).reshape(-1, hkv, bs, d)
    vp = vc.reshape(R, hkv, M // bs, bs, d).transpose(0, 2, 1, 3, 4).reshape(-1, hkv, bs, d)
    layer = _layer(hq, hkv, d, window=w)
    rows, pos = [0, 1], [37, 25]
    q = _rand(2, hq, d)
    want = O.attn_decode_paged(layer, q, kp, vp, table, bs, rows, pos)
    recycled = table.copy()
    for i, p in enumerate(pos):
        first_needed = p - w + 1
        for b in range(M // bs):
            if (b + 1) * bs <= first_needed:
                kp[recycled[rows[i], b]] = np.nan
                recycled[rows[i], b] = -1
    assert (recycled < 0).sum() == 8 + 5
    np.testing.assert_array_equal(O.attn_decode_paged(layer, q, kp, vp, recycled, bs, rows, pos), want)
    bad = recycled.copy()
    bad[0, (pos[0] - w + 1) // bs] = -1                 # the block holding the oldest visible key
    with pytest.raises(ValueError):
        O.attn_decode_paged(layer, q, kp, vp, bad, bs, rows, pos)


def test_paged_update_writes_its_slot_only():
    """The paged update writes what the contiguous update writes at (row, position), at the slot
    (table[row, p // bs], p % bs), and nothing else."""
    hq, hkv, d, bs = 2, 2, 8, 4
    layer = _layer(hq, hkv, d)
    kp, vp = _rand(6, hkv, bs, d), _rand(6, hkv, bs, d)
    k0, v0 = kp.copy(), vp.copy()
    table = np.array([[5, 1, 3], [0, 2, 4]])
    rows, pos = [1, 0], [6, 9]
    q, k, v = _rand(2, hq, d), _rand(2, hkv, d), _rand(2, hkv, d)
    ang = RNG.uniform(-3, 3, (2, d // 2))
    cos, sin = np.cos(ang), np.sin(ang)
    kc, vc = np.zeros((2, hkv, 12, d)), np.zeros((2, hkv, 12, d))
    q_want = O.kv_cache_update(layer, q, k, v, rows, pos, cos, sin, kc, vc)
    q_got = O.kv_cache_update_paged(layer, q, k, v, rows, pos, cos, sin, kp, vp, table, bs)
    np.testing.assert_array_equal(q_got, q_want)
    written = {}
    for r, p in zip(rows, pos):
        written[(table[r, p // bs], p % bs)] = (r, p)
    assert len(written) == 2
    for b in range(6):
        for o in range(bs):
            if (b, o) in written:
                r, p = written[(b, o)]
                np.testing.assert_array_equal(kp[b, :, o], kc[r, :, p])
                np.testing.assert_array_equal(vp[b, :, o], vc[r, :, p])
            else:
                np.testing.assert_array_equal(kp[b, :, o], k0[b, :, o])
                np.testing.assert_array_equal(vp[b, :, o], v0[b, :, o])
