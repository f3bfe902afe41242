"""MLA decode (absorbed form) on the GPU against the oracle: the rows written by the cache update (rotary part
deinterleaved and rotated), the queries' rotated rotary part, and the latent outputs, over contiguous caches
and paged pools; a full-size DeepSeek-V3-shaped step checked on sampled outputs."""
import numpy as np
import pytest
import torch

from oracle import mla as OM

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


def _close(got, ref):
    d = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(d).all()
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())


def _run(call, paged_block=0):
    from decoder_attention_gb300 import _abi, inputs, step
    if paged_block:
        kp, _, table = inputs.paged_from_contiguous(call.cache[:, None], call.cache[:, None], paged_block, seed=4,
                                                    spare_blocks=2)
        st = step.MlaDecodeStep(call, kp, table, paged_block)
    else:
        st = step.MlaDecodeStep(call)
    st.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    return st


@pytest.mark.parametrize("window", [0, 100])
@pytest.mark.parametrize("heads", [16, 128])
def test_mla_decode_matches_oracle(cuda, heads, window):
    from decoder_attention_gb300 import inputs
    call = inputs.deepseek_v3_mla_decode("small")
    if heads != call.num_heads:
        g = torch.Generator().manual_seed(heads)
        call.q = (torch.randn((call.n_seqs, heads, 576), generator=g) * 0.5).to(torch.bfloat16)
        call.num_heads = heads
    call.window = window
    ref = OM.run_mla_call(call)
    st = _run(call.to(cuda))
    _close(st.out, ref["out"])
    # the written rows: latent bit for bit, rotated k_rope within one bf16 rounding
    cache = st.call.cache.cpu()
    for s in range(call.n_seqs):
        r, p = int(call.rows[s]), int(call.positions[s])
        assert torch.equal(cache[r, p, :512], call.latent[s])
        np.testing.assert_allclose(cache[r, p, 512:].double().numpy(), ref["cache"][r, p, 512:], rtol=2.0 ** -8,
                                   atol=1e-6)
    np.testing.assert_allclose(st.q_rot[..., 512:].double().cpu().numpy(), ref["q_rot"][..., 512:], rtol=2.0 ** -8,
                               atol=1e-6)


@pytest.mark.parametrize("block", [64, 128])
def test_mla_decode_paged(cuda, block):
    from decoder_attention_gb300 import inputs
    call = inputs.deepseek_v3_mla_decode("small")
    call.window = 130
    ref = OM.run_mla_call(call)
    st = _run(call.to(cuda), paged_block=block)
    _close(st.out, ref["out"])


def test_mla_full_size_sampled(cuda):
    """The DeepSeek-V3-shaped step (64 sequences up to 32K context, 128 heads): every output row of 6 sampled
    sequences against the oracle on those sequences' own rows."""
    from decoder_attention_gb300 import inputs
    call = inputs.deepseek_v3_mla_decode("full", device=cuda)
    st = _run(call)
    out = st.out.cpu()
    sc = OM.mla_scale(128, 64, call.rope_scaling)
    cpu = call.to("cpu")
    for s in (0, 7, 21, 40, 55, 63):
        sub = inputs.MlaCall(**{k: getattr(cpu, k) for k in cpu.__dataclass_fields__})
        r, p = int(cpu.rows[s]), int(cpu.positions[s])
        sub.q, sub.latent, sub.k_rope = cpu.q[s:s + 1], cpu.latent[s:s + 1], cpu.k_rope[s:s + 1]
        sub.rows, sub.positions, sub.seq_len = torch.tensor([0], dtype=torch.int32), cpu.positions[s:s + 1], cpu.seq_len[s:s + 1]
        sub.cache = cpu.cache[r:r + 1, :p + 1]
        ref = OM.run_mla_call(sub)
        assert abs(OM.mla_scale(128, 64, sub.rope_scaling) - sc) < 1e-15
        _close(out[s:s + 1], ref["out"])
