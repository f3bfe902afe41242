"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the seeded workloads.

Tolerances (stated by the target for this step): bf16 I/O max-abs 2e-2 and mean-abs 2e-3 on the
attention output, fp32 path max-abs 1e-4. Cache bookkeeping is bit-exact: every V slot written equals the
input v, every slot not written keeps its previous bits. q_rot and the K slots are the oracle's rotated
vectors rounded once to bf16 (fp32 arithmetic): within 2^-8 relative plus a small absolute floor.
"""
import numpy as np
import pytest
import torch

from oracle import step as ostep

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP32_MAX = 2e-2, 2e-3, 1e-4


def _run(call, dev):
    from decoder_attention_gb300 import _abi, step
    g = call.to(dev)
    st = step.AttentionStep(g)
    st.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    return st, g


def _check_out(got, ref, fp32):
    diff = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(diff).all()
    if fp32:
        assert diff.max() <= FP32_MAX, diff.max()
    else:
        assert diff.max() <= BF16_MAX, diff.max()
        assert diff.mean() <= BF16_MEAN, diff.mean()
    return diff


def _check_rot(got, ref, fp32):
    g = got.double().cpu().numpy()
    if fp32:
        np.testing.assert_allclose(g, ref, rtol=2e-6, atol=2e-6)
    else:
        np.testing.assert_allclose(g, ref, rtol=2.0 ** -8, atol=1e-6)


def _check_cache(call_cpu, g, ref):
    """Written slots: V bit-exact, K = rotated k within rounding. Others: unchanged bits."""
    rows = call_cpu.tok_rows.numpy()
    pos = call_cpu.tok_pos.numpy()
    kc_after = g.k_cache.cpu()
    vc_after = g.v_cache.cpu()
    written = torch.zeros(call_cpu.k_cache.shape[0], call_cpu.k_cache.shape[2], dtype=torch.bool)
    written[torch.as_tensor(rows, dtype=torch.long), torch.as_tensor(pos, dtype=torch.long)] = True
    w4 = written[:, None, :, None].expand_as(kc_after)
    assert torch.equal(kc_after[~w4], call_cpu.k_cache[~w4])
    assert torch.equal(vc_after[~w4], call_cpu.v_cache[~w4])
    for t in range(len(rows)):
        assert torch.equal(vc_after[rows[t], :, pos[t]], call_cpu.v[t])
    fp32 = call_cpu.dtype == torch.float32
    k_slots = kc_after[torch.as_tensor(rows, dtype=torch.long), :, torch.as_tensor(pos, dtype=torch.long)]
    _check_rot(k_slots, ref["k_cache"][rows, :, pos], fp32)


@pytest.mark.parametrize("number", [1, 2, 3, 4, 5])
def test_small_workload_parity(cuda, number):
    from decoder_attention_gb300 import inputs
    wl = inputs.make(number, scale="small" if number > 1 else "full")
    for call in wl.layers:
        st, g = _run(call, cuda)
        ref = ostep.run_layer_call(call)
        fp32 = call.dtype == torch.float32
        _check_out(st.out, ref["out"], fp32)
        _check_rot(st.q_rot, ref["q_rot"], fp32)
        _check_cache(call, g, ref)
        # cos/sin tables: fp64 angles reduced mod 2 pi, fp32 sine/cosine
        st.rope()                               # the tables themselves (the step may fuse them)
        torch.cuda.synchronize()
        np.testing.assert_allclose(st.cos.cpu().double().numpy(), ref["cos"], atol=5e-7, rtol=0)
        np.testing.assert_allclose(st.sin.cpu().double().numpy(), ref["sin"], atol=5e-7, rtol=0)


def test_softcap_binds(cuda):
    """Workload 5 with q x 8: logits reach ~30 against the cap of 50, so the soft-cap shapes the result. At
    such logits the bf16 rounding of the stored rotated q and k alone moves a logit by ~0.1, which a peaked
    softmax turns into output changes above 2e-2; the attention kernels are therefore checked against the
    oracle with its rotated q/k rounded to bf16 as the cache stores them (the rotation itself is checked
    against the unrounded oracle in the other tests)."""
    from decoder_attention_gb300 import inputs
    wl = inputs.make(5, scale="small", q_mult=8.0)
    for call in wl.layers:
        st, _ = _run(call, cuda)
        ref = ostep.run_layer_call(call, storage_rounding=True)
        _check_out(st.out, ref["out"], False)
        # the cap binds: the uncapped result differs grossly
        import copy
        nocap = copy.copy(call)
        nocap.softcap = 0.0
        ref_nocap = ostep.run_layer_call(nocap, storage_rounding=True)
        assert np.abs(ref_nocap["out"] - ref["out"]).max() > 0.1


def test_softcap_binds_against_unrounded_oracle(cuda):
    """Workload 5 with q x 1.75 against the exact (unrounded) fp64 oracle at the standard bf16 tolerance,
    with the cap binding: removing it moves the oracle's outputs by more than 0.05. Measured on GB300: the
    largest q multiple inside the tolerance is about 1.9 (max error 0.017); at 2 the bf16 storage of the
    rotated q and k alone takes the max error to 0.021."""
    from decoder_attention_gb300 import inputs
    import copy
    wl = inputs.make(5, scale="small", q_mult=1.75)
    for call in wl.layers:
        st, _ = _run(call, cuda)
        ref = ostep.run_layer_call(call)
        _check_out(st.out, ref["out"], False)
        nocap = copy.copy(call)
        nocap.softcap = 0.0
        assert np.abs(ostep.run_layer_call(nocap)["out"] - ref["out"]).max() > 0.05


def test_repeat_is_deterministic(cuda):
    """Two runs on the same inputs give bit-identical outputs (fixed merge order, no atomics)."""
    from decoder_attention_gb300 import inputs
    call = inputs.make(3, scale="small").layers[0]
    st1, _ = _run(call, cuda)
    st2, _ = _run(call, cuda)
    assert torch.equal(st1.out, st2.out)
