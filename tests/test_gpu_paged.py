"""Paged KV pool on the GPU against the oracle's paged functions: the cache update writes through the block
table, prefill and decode read through it, with blocks in random pool order, spare blocks, and (for windowed
layers) the blocks before every query's window unmapped and filled with NaN, as a pool that recycles them
leaves them. Block sizes that are multiples of 64 run the tensor-core kernels; others the CUDA-core kernel."""
import numpy as np
import pytest
import torch

from oracle import step as ostep

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP32_MAX = 2e-2, 2e-3, 1e-4


def _close(got, ref, fp32=False):
    d = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(d).all()
    if fp32:
        assert d.max() <= FP32_MAX, d.max()
    else:
        assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())


def _first_needed(call):
    """Per cache row, the oldest position any token of the call can see (blocks wholly before it are unused)."""
    R = call.num_rows
    need = np.full(R, 0 if not call.window else np.iinfo(np.int64).max, dtype=np.int64)
    if call.window:
        for r, p in zip(call.tok_rows.tolist(), call.tok_pos.tolist()):
            need[r] = min(need[r], max(0, p - call.window + 1))
        if call.n_prefill:
            starts = call.q_start.tolist()
            for b, (r, fp) in enumerate(zip(call.pf_rows.tolist(), call.pf_first_pos.tolist())):
                if starts[b + 1] > starts[b]:
                    need[r] = min(need[r], max(0, fp - call.window + 1))
        need[need == np.iinfo(np.int64).max] = 0
    return need


def _row_ends(call):
    """Per cache row, one past the last position the call writes or reads (blocks from there on are unused)."""
    end = np.zeros(call.num_rows, dtype=np.int64)
    for r, p in zip(call.tok_rows.tolist(), call.tok_pos.tolist()):
        end[r] = max(end[r], p + 1)
    return end


def _run_paged(call, cuda, block_size, seed, recycle):
    from decoder_attention_gb300 import _abi, inputs, step
    g = call.to(cuda)
    unmap = _first_needed(call) if recycle else None
    ends = _row_ends(call) if recycle else None
    kp, vp, table = inputs.paged_from_contiguous(g.k_cache, g.v_cache, block_size, seed=seed, spare_blocks=3,
                                                 unmap_before=unmap, unmap_from=ends)
    ref = ostep.run_layer_call_paged(call, kp.cpu(), vp.cpu(), table.cpu(), block_size)
    st = step.PagedAttentionStep(g, kp, vp, table, block_size)
    st.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    return st, ref


def _layers(workload):
    from decoder_attention_gb300 import inputs
    return inputs.make(workload, "small").layers


@pytest.mark.parametrize("block_size", [64, 128, 256, 16])
@pytest.mark.parametrize("workload", ["qwen3_8b_prefill", "mistral_swa_decode", "phi4_gemma2_mixed"])
def test_paged_step_matches_oracle(cuda, workload, block_size):
    for li, call in enumerate(_layers(workload)):
        st, ref = _run_paged(call, cuda, block_size, seed=li + block_size, recycle=True)
        _close(st.out[:call.n_tokens], ref["out"])
        # the pools after the update: V slots bit for bit, K within one bf16 rounding, the rest untouched
        table = st.block_table.cpu().numpy()
        vp = st.v_pool.cpu()
        for t, (r, p) in enumerate(zip(call.tok_rows.tolist(), call.tok_pos.tolist())):
            b = table[r, p // block_size]
            assert torch.equal(vp[b, :, p % block_size], call.v[t])
        kp = st.k_pool.double().cpu().numpy()
        mapped = table[table >= 0]
        np.testing.assert_allclose(kp[mapped], ref["k_pool"][mapped], rtol=2.0 ** -8, atol=1e-6)


def test_paged_fp32_and_sinks(cuda):
    """The fp32 path (CUDA-core kernel) over a paged pool, with learned sinks."""
    call = _layers("tiny_prefill_fp32")[0]
    call.sinks = torch.tensor([0.5, -1.0, 2.0, -30.0])
    st, ref = _run_paged(call, cuda, 32, seed=3, recycle=False)
    _close(st.out, ref["out"], fp32=True)


def test_unmapped_visible_block_is_reported(cuda):
    """A visible position whose block is unmapped sets the device error word (no fault; its keys are not the
    caller's)."""
    from decoder_attention_gb300 import _abi, inputs, step
    call = _layers("mistral_swa_decode")[0].to(cuda)
    kp, vp, table = inputs.paged_from_contiguous(call.k_cache, call.v_cache, 64, seed=9)
    r, p = int(call.dec_rows[0]), int(call.dec_pos[0])
    table[r, p // 64] = -1                                  # the block of the token's own position
    st = step.PagedAttentionStep(call, kp, vp, table, 64)
    st.run()
    torch.cuda.synchronize()
    with pytest.raises(_abi.DecAttnError) as ei:
        _abi.check_device_error()
    assert ei.value.code == _abi.DA_ERR_DEVICE_INDEX


def test_pool_recycling_over_many_steps(cuda):
    """A serving loop over one paged pool: four requests prefill, then decode one token per step while the
    block manager recycles the blocks that fall out of their 128-key window (and hands them to other
    requests); a finished request's row is released and reused by a new request. Every step's output is
    checked against the oracle over contiguous caches holding the same history."""
    import math
    from decoder_attention_gb300 import _abi, inputs, step
    from oracle import attention as A
    hq, hkv, d, w, bs, R = 8, 2, 128, 128, 64, 4
    max_blocks = 16                                     # rows hold up to 1024 positions
    n_blocks = R * (math.ceil(w / bs) + 1) + 8           # far fewer than R * max_blocks: recycling is required
    pool = _abi.BlockPool(n_blocks, bs, R, max_blocks, window=w)
    kp = torch.full((n_blocks, hkv, bs, d), float("nan"), dtype=torch.bfloat16, device=cuda)
    vp = torch.full_like(kp, float("nan"))
    g = torch.Generator().manual_seed(77)
    layer = A.Layer(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, rotary_dim=d, window=w)
    kc = np.zeros((R, hkv, max_blocks * bs, d))
    vc = np.zeros_like(kc)
    length = [0] * R

    def run_step(rows, positions, n_prefill, q_start=None, first_pos=None, max_q_len=0):
        n = len(rows)
        q = (torch.randn((n, hq, d), generator=g) / math.sqrt(d) * 4).to(torch.bfloat16)
        k = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
        v = torch.randn((n, hkv, d), generator=g).to(torch.bfloat16)
        seq_len = [max(positions[j] + 1 for j in range(n) if rows[j] == r) for r in rows]
        dec_rows, dec_pos = rows[n_prefill:], positions[n_prefill:]
        call = inputs.LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv,
                                partial_rotary_factor=1.0, rope_theta=1e4, rope_scaling=None,
                                max_position_embeddings=max_blocks * bs, dtype=torch.bfloat16, window=w,
                                q=q, k=k, v=v, tok_rows=inputs._i32(rows), tok_pos=inputs._i32(positions),
                                tok_seq_len=inputs._i32(seq_len), n_prefill=n_prefill,
                                q_start=inputs._i32(q_start or [0]), pf_rows=inputs._i32(sorted(set(rows[:n_prefill]),
                                key=rows.index) if n_prefill else []),
                                pf_first_pos=inputs._i32(first_pos or []), max_q_len=max_q_len,
                                dec_rows=inputs._i32(dec_rows), dec_pos=inputs._i32(dec_pos),
                                k_cache=torch.empty(R, hkv, 1, d, dtype=torch.bfloat16),
                                v_cache=torch.empty(R, hkv, 1, d, dtype=torch.bfloat16))
        table = pool.table().to(cuda)
        st = step.PagedAttentionStep(call.to(cuda), kp, vp, table, bs)
        st.run()
        torch.cuda.synchronize()
        _abi.check_device_error()
        # oracle on contiguous caches with the same history
        cos, sin = A.rope_tables_for_tokens(A.RopeSpec(theta=1e4), d, positions)
        q_rot = A.kv_cache_update(layer, q.double().numpy(), k.double().numpy(), v.double().numpy(), rows,
                                  positions, cos, sin, kc, vc)
        want = np.zeros_like(q_rot)
        if n_prefill:
            want[:n_prefill] = A.attn_prefill(layer, q_rot[:n_prefill], kc, vc, q_start, call.pf_rows.tolist(),
                                              first_pos)
        if n > n_prefill:
            want[n_prefill:] = A.attn_decode(layer, q_rot[n_prefill:], kc, vc, dec_rows, dec_pos)
        _close(st.out, want)

    def prefill(r, n):
        pool.reserve(r, 0, n)
        run_step([r] * n, list(range(n)), n, [0, n], [0], n)
        length[r] = n

    for r, n in enumerate([200, 150, 300, 90]):
        prefill(r, n)
    for s in range(120):
        if s == 60:                                      # request 1 finishes; a new one takes its row
            pool.release(1)
            kc[1] = 0.0
            vc[1] = 0.0
            prefill(1, 170)
        rows = list(range(R))
        pos = [length[r] for r in rows]
        for r in rows:
            pool.reserve(r, length[r], length[r] + 1)
        run_step(rows, pos, 0)
        for r in rows:
            length[r] += 1
    assert max(length) > n_blocks * bs // R             # the rows outgrew their share without recycling
