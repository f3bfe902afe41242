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


def _run_paged(call, cuda, block_size, seed, recycle):
    from decoder_attention_gb300 import _abi, inputs, step
    g = call.to(cuda)
    unmap = _first_needed(call) if recycle else None
    kp, vp, table = inputs.paged_from_contiguous(g.k_cache, g.v_cache, block_size, seed=seed, spare_blocks=3,
                                                 unmap_before=unmap)
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
