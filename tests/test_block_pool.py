"""The paged pool's host block manager (da_block_pool, native, no GPU): invariants under random use, the
all-or-nothing reserve, recycling of out-of-window blocks, and the page's bound of ceil(w / block) + 1
blocks per windowed-only request (page 1, "Sliding windows"), with the Mistral question it poses: how many
more 32K-context requests fit in one pool when out-of-window blocks are recycled."""
import math

import numpy as np
import pytest

_abi = pytest.importorskip("decoder_attention_gb300._abi",
                           reason="libdecattn.so not built (run __graft_entry__.build())")


def _check_invariants(pool, state):
    t = pool.table().numpy()
    ids = t[t >= 0]
    assert len(ids) == len(set(ids.tolist())), "a block is mapped twice"
    assert ((ids >= 0) & (ids < pool.n_blocks)).all()
    assert pool.free_blocks + len(ids) == pool.n_blocks
    for r in range(pool.num_rows):
        if r not in state:
            assert (t[r] < 0).all()
            continue
        first_pos, length = state[r]
        lo = max(0, first_pos - pool.window + 1) if pool.window else 0
        want = set(range(lo // pool.block_size, math.ceil(length / pool.block_size)))
        assert set(np.nonzero(t[r] >= 0)[0].tolist()) == want, (r, first_pos, length)


@pytest.mark.parametrize("window,bs", [(0, 16), (50, 16), (64, 64), (7, 4)])
def test_random_use_keeps_the_table_consistent(window, bs):
    rng = np.random.default_rng(window + bs)
    R, max_blocks = 6, 40
    pool = _abi.BlockPool(120, bs, R, max_blocks, window)
    state = {}
    for _ in range(400):
        r = int(rng.integers(R))
        op = rng.random()
        if op < 0.1 and r in state:
            pool.release(r)
            del state[r]
        else:
            first, length = state.get(r, (0, 0))
            new_first = length                         # this step's oldest query: the row's next token
            new_len = min(length + int(rng.integers(1, 3 * bs)), max_blocks * bs)
            if new_len <= new_first:
                continue
            before = pool.table().clone()
            free = pool.free_blocks
            try:
                pool.reserve(r, new_first, new_len)
                state[r] = (new_first, new_len)
            except _abi.DecAttnError as e:
                assert e.code == _abi.DA_ERR_OUT_OF_BLOCKS
                assert (pool.table() == before).all() and pool.free_blocks == free   # all or nothing
        _check_invariants(pool, state)


def test_recycled_block_is_handed_out_next():
    pool = _abi.BlockPool(10, 4, 2, 8, window=6)
    pool.reserve(0, 0, 5)                      # positions 0..4: blocks 0, 1
    t = pool.table()
    assert t[0, :2].tolist() == [0, 1]
    pool.reserve(0, 9, 10)                     # query at 9 sees 4..9: block index 0 goes back to the pool
    t = pool.table()
    assert t[0, 0] == -1 and t[0, 1] == 1 and t[0, 2] == 0


def test_out_of_blocks_and_bad_arguments():
    pool = _abi.BlockPool(3, 8, 2, 4)
    pool.reserve(0, 0, 16)
    with pytest.raises(_abi.DecAttnError) as e:
        pool.reserve(1, 0, 17)                 # needs 3 blocks, 1 free
    assert e.value.code == _abi.DA_ERR_OUT_OF_BLOCKS
    for args in ((2, 0, 1), (0, -1, 1), (0, 5, 4), (0, 0, 33)):
        with pytest.raises(_abi.DecAttnError) as e:
            pool.reserve(*args)
        assert e.value.code == _abi.DA_ERR_INVALID_ARG
    pool.release(0)
    assert pool.free_blocks == 3
    pool.reserve(1, 0, 17)


@pytest.mark.parametrize("w,bs", [(4096, 64), (4096, 16), (1000, 64), (128, 128)])
def test_windowed_request_holds_at_most_w_over_block_plus_one(w, bs):
    """Page 1: a model with only windowed layers needs ceil(w / block size) + 1 blocks per request."""
    pool = _abi.BlockPool(10_000, bs, 1, 70_000 // bs + 1, window=w)
    bound = math.ceil(w / bs) + 1
    most = 0
    for p in range(0, 70_000, 97):             # one decode step at a time (every 97th position)
        pool.reserve(0, p, p + 1)
        most = max(most, 10_000 - pool.free_blocks)
    assert most == bound


def test_mistral_requests_at_32k_context():
    """The page's question for Mistral 7B (window 4096) at 32K context: requests that fit in one pool with and
    without recycling the out-of-window blocks (64-position blocks, 4096 blocks in the pool)."""
    bs, n_blocks, ctx = 64, 4096, 32768

    def admitted(window):
        pool = _abi.BlockPool(n_blocks, bs, 256, ctx // bs, window=window)
        n = 0
        while True:
            try:
                pool.reserve(n, ctx - 18, ctx - 17)   # a request decoding near 32K, its window starting mid-block
            except _abi.DecAttnError:
                return n
            n += 1

    full, windowed = admitted(0), admitted(4096)
    assert full == n_blocks // (ctx // bs) == 8
    assert windowed == n_blocks // (4096 // bs + 1) == 63     # 65 blocks each: 7.9 times as many requests
