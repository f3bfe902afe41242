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


def _close_scaled(got, ref):
    """_close relative to the output's magnitude: bf16 rounding of the rotated queries and of the new row is
    relative, so with rows scaled well above 1 (outputs up to ~40) the absolute error grows with them."""
    scale = max(1.0, float(np.abs(ref).max()))
    _close(got.double() / scale, ref / scale)


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


def _sub_call(cpu, s):
    """Sequence s of a call alone (its own row and visible positions), for the oracle."""
    from decoder_attention_gb300 import inputs
    sub = inputs.MlaCall(**{k: getattr(cpu, k) for k in cpu.__dataclass_fields__})
    r, p = int(cpu.rows[s]), int(cpu.positions[s])
    sub.q, sub.latent, sub.k_rope = cpu.q[s:s + 1], cpu.latent[s:s + 1], cpu.k_rope[s:s + 1]
    sub.rows, sub.positions, sub.seq_len = torch.tensor([0], dtype=torch.int32), cpu.positions[s:s + 1], cpu.seq_len[s:s + 1]
    sub.cache = cpu.cache[r:r + 1, :p + 1]
    return sub


@pytest.mark.parametrize("block", [0, 64, 256])
@pytest.mark.parametrize("window", [0, 1000])
def test_mla_128_heads_multi_tile_rescale(cuda, window, block):
    """128 heads (the CTA-pair kernel) with chunks of several 256-key tiles: 40 sequences of up to 4096 keys
    (512-key chunks), lengths at and around the tile and chunk edges, rows whose scale grows with position so
    that the running max moves (and O is rescaled) on many tiles, and NaN in every slot past a sequence's new
    token; contiguous and paged pools; sampled sequences, every head, against the oracle."""
    from decoder_attention_gb300 import inputs
    S, M, H = 40, 4096, 128
    g = torch.Generator().manual_seed(77 + window)
    lens = [4096, 4095, 3841, 3840, 2049, 1025, 513, 512, 257, 256, 255, 1]
    lens += torch.randint(1, M + 1, (S - len(lens),), generator=g).tolist()
    ramp = 1.0 + torch.arange(M, dtype=torch.float32) / 512.0
    cache = (torch.randn((S, M, 576), generator=g) * ramp[None, :, None]).to(torch.bfloat16)
    rows = torch.randperm(S, generator=g).to(torch.int32)
    for s, n in enumerate(lens):   # never-written slots past each sequence's new token: they must not matter
        cache[int(rows[s]), n:] = float("nan")
    call = inputs.MlaCall(num_heads=H, qk_nope_head_dim=128, qk_rope_head_dim=64, rope_theta=1e4,
                          rope_scaling=inputs.DEEPSEEK_V3_YARN, max_position_embeddings=163840,
                          q=(torch.randn((S, H, 576), generator=g) * 0.5).to(torch.bfloat16),
                          latent=torch.randn((S, 512), generator=g).to(torch.bfloat16),
                          k_rope=torch.randn((S, 64), generator=g).to(torch.bfloat16), rows=rows,
                          positions=torch.tensor([n - 1 for n in lens], dtype=torch.int32),
                          seq_len=torch.tensor(lens, dtype=torch.int32), cache=cache, window=window)
    st = _run(call.to(cuda), paged_block=block)
    out = st.out.cpu()
    for s in (0, 1, 2, 5, 7, 9, 10, 11):
        _close_scaled(out[s:s + 1], OM.run_mla_call(_sub_call(call, s))["out"])


@pytest.mark.parametrize("heads", [16, 128])
def test_mla_invalid_sequence(cuda, heads):
    """A sequence whose cache row is out of range: the device error word says so, its outputs are zero and the
    other sequences are unaffected (legacy and CTA-pair kernels)."""
    from decoder_attention_gb300 import _abi, inputs
    call = inputs.deepseek_v3_mla_decode("small")
    if heads != call.num_heads:
        g = torch.Generator().manual_seed(heads)
        call.q = (torch.randn((call.n_seqs, heads, 576), generator=g) * 0.5).to(torch.bfloat16)
        call.num_heads = heads
    good = call.to("cpu")
    bad = inputs.MlaCall(**{k: getattr(call, k) for k in call.__dataclass_fields__})
    bad.rows = call.rows.clone()
    bad.rows[1] = call.num_rows                      # one past the last row
    from decoder_attention_gb300 import step
    st = step.MlaDecodeStep(bad.to(cuda))
    st.run()
    torch.cuda.synchronize()
    with pytest.raises(_abi.DecAttnError) as ei:
        _abi.check_device_error()
    assert ei.value.code == _abi.DA_ERR_DEVICE_INDEX
    out = st.out.cpu()
    assert torch.count_nonzero(out[1]) == 0
    for s in (0, 2, 3, 4):
        _close(out[s:s + 1], OM.run_mla_call(_sub_call(good, s))["out"])
    _abi.check_device_error()                         # the word was cleared
