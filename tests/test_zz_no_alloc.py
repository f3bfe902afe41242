"""da_attn_decode_noalloc: the decode entry point for callers that may not allocate device memory.

It runs the same split-K decode as da_attn_decode but keeps its partial results in the library's fixed
scratch array instead of a caller-provided workspace. The test calls it through the C ABI twice in a row,
on two different decode batches (different split plans, so the second call finds the first call's partials
in the shared scratch). Both entry points run the same kernels with the same split plan and a fixed merge
order, so each result must equal da_attn_decode's on the same inputs bit for bit; the sliding-window batch is
also checked against the fp64 oracle within the bf16 tolerance the parity tests use. This file is collected
last so that a failure here cannot hide the other tests' results; it passes alone in a fresh process and after
the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


def _decode_both(call, dev):
    from decoder_attention_gb300 import _abi, step
    st = step.AttentionStep(call.to(dev))
    st.rope()
    st.cache_update()
    c = st.call
    npf = c.n_prefill
    q = st.q_rot[npf:]
    out_ws = torch.full_like(q, float("nan"))
    out_na = torch.full_like(q, float("nan"))
    _abi.attn_decode(st.L, q, c.k_cache, c.v_cache, c.num_rows, c.max_len, c.n_decode, c.dec_rows, c.dec_pos, None,
                     out_ws, st.workspace, st.ws_bytes)
    _abi.attn_decode_noalloc(st.L, q, c.k_cache, c.v_cache, c.num_rows, c.max_len, c.n_decode, c.dec_rows,
                             c.dec_pos, None, out_na)
    torch.cuda.synchronize()
    _abi.check_device_error()
    return out_ws, out_na, st


def test_noalloc_matches_workspace_decode_twice(cuda):
    from decoder_attention_gb300 import inputs
    from oracle import step as ostep
    first = inputs.make(4, scale="small").layers[0]     # long-context rows, full attention
    second = inputs.make(3, scale="small").layers[0]    # sliding-window rows, other split plan
    for call in (first, second):
        ref, got, st = _decode_both(call, cuda)
        assert st.workspace is not None and st.ws_bytes > 0      # the fast split-K path is the one compared
        assert torch.isfinite(got).all()
        assert torch.equal(got, ref)                             # same kernels, same plan, fixed merge order
    want = ostep.run_layer_call(second)["out"][second.n_prefill:]
    diff = np.abs(got.double().cpu().numpy() - want)
    assert diff.max() <= BF16_MAX and diff.mean() <= BF16_MEAN


def test_noalloc_rejects_plans_beyond_its_scratch(cuda):
    """A batch whose split plan needs more than the fixed scratch is refused before any work is enqueued."""
    from decoder_attention_gb300 import _abi
    L = _abi.layer(torch.bfloat16, 128, 64, 8, 128)
    n_seqs, max_len = 4096, 131072
    assert _abi.decode_workspace_bytes(L, n_seqs, max_len) > _abi.decode_noalloc_max_scratch_bytes()
    d = ctypes.c_void_p(256)
    rc = _abi.LIB.da_attn_decode_noalloc(ctypes.byref(L), d, d, d, 8, max_len, n_seqs, d, d, None, d, None)
    assert rc == _abi.DA_ERR_INVALID_ARG
    assert "scratch" in _abi.last_error()
