"""Edge cases of the CUDA path against the fp64 oracle (through the C ABI).

Covers: calls with nothing to do; a window of one key; a window at least as long as the context, which must
reproduce full attention bit for bit; cache slots past a row's length filled with NaN (they must never
reach a result); explicit key positions (slots permuted); fp32 decode; layers the fast kernels leave to the
CUDA-core kernel (d = 64 in bf16, a GQA group of 16); and out-of-range rows, which the kernels skip and
report through the device error word instead of faulting.
"""
import copy
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import step as ostep

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, FP32_MAX = 2e-2, 2e-3, 1e-4


def _abi():
    from decoder_attention_gb300 import _abi
    return _abi


def _run(call, dev):
    from decoder_attention_gb300 import step
    g = call.to(dev)
    st = step.AttentionStep(g)
    st.run()
    torch.cuda.synchronize()
    _abi().check_device_error()
    return st, g


def _close(got, ref, fp32=False):
    d = np.abs(got.double().cpu().numpy() - ref)
    assert np.isfinite(d).all()
    if fp32:
        assert d.max() <= FP32_MAX, d.max()
    else:
        assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())


def _prefill_call(lens, first_pos, hq=8, hkv=2, d=128, window=0, softcap=0.0, dtype=torch.bfloat16, seed=5,
                  M=None, rot=None, sinks=None, rope_scaling=None, theta=1e4, max_pos=None):
    """A prefill-only call with random caches for the positions before each chunk."""
    from decoder_attention_gb300 import inputs
    g = torch.Generator().manual_seed(seed)
    n = sum(lens)
    q = (torch.randn((n, hq, d), generator=g) / math.sqrt(d) * 4).to(dtype)
    k = torch.randn((n, hkv, d), generator=g).to(dtype)
    v = torch.randn((n, hkv, d), generator=g).to(dtype)
    R = len(lens)
    M = M or max(p + L for p, L in zip(first_pos, lens))
    kc = torch.randn((R, hkv, M, d), generator=g).to(dtype)
    vc = torch.randn((R, hkv, M, d), generator=g).to(dtype)
    qs, tr, tp, tl = inputs._prefill_meta(lens, first_pos, list(range(R)))
    return inputs.LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv,
                            partial_rotary_factor=(rot or d) / d, rope_theta=theta, rope_scaling=rope_scaling,
                            max_position_embeddings=max_pos or M, dtype=dtype, window=window, softcap=softcap,
                            sinks=sinks,
                            q=q, k=k, v=v, tok_rows=inputs._i32(tr), tok_pos=inputs._i32(tp),
                            tok_seq_len=inputs._i32(tl), n_prefill=n, q_start=inputs._i32(qs),
                            pf_rows=inputs._i32(list(range(R))), pf_first_pos=inputs._i32(first_pos),
                            max_q_len=max(lens), dec_rows=inputs._i32([]), dec_pos=inputs._i32([]),
                            k_cache=kc, v_cache=vc)


def _decode_call(lens, hq=8, hkv=2, d=128, window=0, dtype=torch.bfloat16, seed=6, sinks=None, softcap=0.0):
    from decoder_attention_gb300 import inputs
    g = torch.Generator().manual_seed(seed)
    S = len(lens)
    M = max(lens)
    q = (torch.randn((S, hq, d), generator=g) / math.sqrt(d) * 4).to(dtype)
    k = torch.randn((S, hkv, d), generator=g).to(dtype)
    v = torch.randn((S, hkv, d), generator=g).to(dtype)
    kc = torch.randn((S, hkv, M, d), generator=g).to(dtype)
    vc = torch.randn((S, hkv, M, d), generator=g).to(dtype)
    pos = [L - 1 for L in lens]
    rows = list(range(S))
    return inputs.LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, partial_rotary_factor=1.0,
                            rope_theta=1e4, rope_scaling=None, max_position_embeddings=M, dtype=dtype,
                            window=window, softcap=softcap, sinks=sinks, q=q, k=k, v=v, tok_rows=inputs._i32(rows), tok_pos=inputs._i32(pos),
                            tok_seq_len=inputs._i32(lens), n_prefill=0, q_start=inputs._i32([0]),
                            pf_rows=inputs._i32([]), pf_first_pos=inputs._i32([]), max_q_len=0,
                            dec_rows=inputs._i32(rows), dec_pos=inputs._i32(pos), k_cache=kc, v_cache=vc)


def test_empty_calls_do_nothing(cuda):
    ab = _abi()
    L = ab.layer(torch.bfloat16, 128, 8, 2, 128)
    x = torch.zeros(16, dtype=torch.bfloat16, device=cuda)
    i = torch.zeros(4, dtype=torch.int32, device=cuda)
    f = torch.zeros(16, dtype=torch.float32, device=cuda)
    rs, keep = ab.rope_scaling(1e4, 128)
    ab.rope_tables_build(rs, i, None, 0, f, f)
    ab.kv_cache_update(L, x, x, x, 0, i, i, f, f, x, x, x, 1, 1)
    ab.attn_prefill(L, x, 0, x, x, 1, 1, 0, i, i, i, 0, None, x)
    ab.attn_decode(L, x, x, x, 1, 1, 0, i, i, None, x, None, 0)
    torch.cuda.synchronize()
    ab.check_device_error()
    assert torch.count_nonzero(x) == 0


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_window_one_and_window_covering_context(cuda, kind):
    base = (_prefill_call([300, 129], [0, 170]) if kind == "prefill" else _decode_call([700, 1, 129, 4096]))
    one = copy.copy(base)
    one.window = 1
    st, _ = _run(one, cuda)
    _close(st.out, ostep.run_layer_call(one)["out"])
    full, _ = _run(base, cuda)
    wide = copy.copy(base)
    wide.window = 1 << 20
    st_w, _ = _run(wide, cuda)
    assert torch.equal(st_w.out, full.out)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_nan_in_unwritten_slots_never_reaches_the_result(cuda, kind):
    call = _prefill_call([77, 200], [0, 333]) if kind == "prefill" else _decode_call([65, 1000, 3, 130])
    ref = ostep.run_layer_call(call)["out"]
    poisoned = copy.copy(call)
    kc, vc = call.k_cache.clone(), call.v_cache.clone()
    if kind == "prefill":
        ends = [p + L for p, L in zip(call.pf_first_pos.tolist(), np.diff(call.q_start.numpy()).tolist())]
        rows = call.pf_rows.tolist()
    else:
        ends = [p + 1 for p in call.dec_pos.tolist()]
        rows = call.dec_rows.tolist()
    for r, e in zip(rows, ends):
        kc[r, :, e:] = float("nan")
        vc[r, :, e:] = float("nan")
    poisoned.k_cache, poisoned.v_cache = kc, vc
    st, _ = _run(poisoned, cuda)
    _close(st.out, ref)


def test_explicit_key_positions(cuda):
    """With key_positions the mask compares positions: a row whose slots are permuted (positions alike)
    gives the oracle's result; -1 marks empty slots (filled with NaN here)."""
    ab = _abi()
    from decoder_attention_gb300 import step
    call = _prefill_call([150], [90], window=64)
    ref = ostep.run_layer_call(call)["out"]
    st = step.AttentionStep(call.to(cuda))
    st.rope()
    st.cache_update()
    torch.cuda.synchronize()
    M = call.k_cache.shape[2]
    kv_len = 90 + 150
    perm = torch.randperm(kv_len, generator=torch.Generator().manual_seed(3))
    kp = torch.full((1, M + 8), -1, dtype=torch.int32)
    kp[0, :kv_len] = perm.to(torch.int32)
    kc = torch.full((1, 2, M + 8, 128), float("nan"), dtype=torch.bfloat16, device=cuda)
    vc = torch.full_like(kc, float("nan"))
    kc[0, :, :kv_len] = st.call.k_cache[0, :, perm.to(cuda)]
    vc[0, :, :kv_len] = st.call.v_cache[0, :, perm.to(cuda)]
    out = torch.empty_like(st.q_rot)
    c = st.call
    ab.attn_prefill(st.L, st.q_rot, c.n_prefill, kc, vc, 1, M + 8, 1, c.q_start, c.pf_rows, c.pf_first_pos,
                    c.max_q_len, kp.to(cuda), out)
    torch.cuda.synchronize()
    ab.check_device_error()
    _close(out, ref)


def test_fp32_decode_and_generic_fallbacks(cuda):
    """fp32 decode (CUDA-core kernel at 1e-4), bf16 d = 64 and a GQA group of 16 (also the CUDA-core kernel)."""
    c32 = _decode_call([40, 1, 513], dtype=torch.float32)
    st, _ = _run(c32, cuda)
    _close(st.out, ostep.run_layer_call(c32)["out"], fp32=True)
    c64 = _prefill_call([100, 33], [0, 50], hq=4, hkv=2, d=64)
    st, _ = _run(c64, cuda)
    _close(st.out, ostep.run_layer_call(c64)["out"])
    g16 = _decode_call([300, 2], hq=16, hkv=1)
    st, _ = _run(g16, cuda)
    _close(st.out, ostep.run_layer_call(g16)["out"])


def test_out_of_range_rows_are_reported_not_faulted(cuda):
    ab = _abi()
    from decoder_attention_gb300 import step
    for call in (_decode_call([50, 60]), _prefill_call([40, 30], [0, 10])):
        g = call.to(cuda)
        st = step.AttentionStep(g)
        st.rope()
        st.cache_update()
        torch.cuda.synchronize()
        ab.check_device_error()
        bad = g.dec_rows.clone() if call.n_decode else g.pf_rows.clone()
        bad[1] = 9999
        if call.n_decode:
            g.dec_rows = bad
            st.decode()
            rows_out = st.out[1]
        else:
            g.pf_rows = bad
            st.prefill()
            qs = g.q_start.tolist()
            rows_out = st.out[qs[1]:qs[2]]
        torch.cuda.synchronize()
        with pytest.raises(ab.DecAttnError) as ei:
            ab.check_device_error()
        assert ei.value.code == ab.DA_ERR_DEVICE_INDEX
        assert torch.count_nonzero(rows_out) == 0          # the bad sequence's outputs are zero
        ab.check_device_error()                             # the word was cleared


def test_rope_tables_at_long_positions(cuda):
    """cos/sin at positions up to 2^17 against fp64 (llama3 scaling and LongRoPE's long table)."""
    ab = _abi()
    pos = torch.tensor([0, 1, 4095, 4096, 8191, 65535, 100003, 131071], dtype=torch.int32)
    for theta, sc, r, mpe in ((5e5, {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0,
                                     "high_freq_factor": 4.0, "original_max_position_embeddings": 8192}, 128, 131072),
                              (1e4, {"rope_type": "longrope", "short_factor": list(np.linspace(1, 1.2, 48)),
                                     "long_factor": list(np.linspace(1, 40, 48)),
                                     "original_max_position_embeddings": 4096}, 96, 131072)):
        rs, keep = ab.rope_scaling(theta, r, sc, mpe)
        lens = pos + 1
        cos = torch.empty((len(pos), r // 2), dtype=torch.float32, device=cuda)
        sin = torch.empty_like(cos)
        ab.rope_tables_build(rs, pos.to(cuda), lens.to(cuda), len(pos), cos, sin)
        torch.cuda.synchronize()
        ab.check_device_error()
        spec = A.RopeSpec(theta=theta, scaling=sc, max_position_embeddings=mpe)
        rc, rsn = A.rope_tables_for_tokens(spec, r, pos.numpy(), lens.numpy())
        np.testing.assert_allclose(cos.cpu().double().numpy(), rc, atol=5e-7, rtol=0)
        np.testing.assert_allclose(sin.cpu().double().numpy(), rsn, atol=5e-7, rtol=0)


@pytest.mark.parametrize("window", [0, 96])
def test_short_chunks_after_a_long_one(cuda, window):
    """A long chunk then twenty chunks too short for a second query tile: the warpgroup of the second tile
    finishes its only item early and then has nothing to do for a long run of items (its finished item must
    not hold the item ring meanwhile); a window makes the two tiles of an item start on different key tiles."""
    lens = [300] + [50] * 20
    fps = [0] + [37 * i for i in range(1, 21)]
    call = _prefill_call(lens, fps, hq=4, hkv=2, window=window, seed=13)
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref)


@pytest.mark.parametrize("heads", [(4, 2), (3, 1), (2, 2)])
@pytest.mark.parametrize("window", [0, 300])
def test_mixed_lengths_and_offsets(cuda, window, heads):
    """Chunks whose work differs widely (lengths 1 to 700, first positions 0 to 1500): the items are handed out
    by their key-tile count, not by chunk order, with ties and chunks too short for the later query tiles.
    Query heads per KV head 2 (items pair two heads on the same rows), 3 and 1 (items pair two row tiles of
    one head)."""
    lens = [40, 700, 130, 513, 1, 256, 257, 600]
    fps = [900, 0, 1300, 17, 1500, 600, 333, 450]
    call = _prefill_call(lens, fps, hq=heads[0], hkv=heads[1], window=window, seed=21)
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref)


def test_more_chunk_tiles_than_the_schedule_table(cuda):
    """520 chunks of one query tile each: more (chunk, query tile) pairs than the cost ranking holds, so the
    items go out in chunk order."""
    g = torch.Generator().manual_seed(3)
    lens = torch.randint(1, 6, (520,), generator=g).tolist()
    fps = torch.randint(0, 100, (520,), generator=g).tolist()
    call = _prefill_call(lens, fps, hq=2, hkv=1, seed=22)
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref)


def _sinks(hq, seed):
    """Learned sink logits for hq heads: N(0, 2) with one far above every score and one far below."""
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(hq, generator=g) * 2
    s[0] = 30.0
    s[-1] = -40.0
    return s


@pytest.mark.parametrize("window,cap", [(0, 0.0), (200, 0.0), (0, 30.0)])
def test_prefill_with_sinks(cuda, window, cap):
    """Learned sinks on the tensor-core prefill: one extra logit per head whose share reaches no value,
    with a window (the sink is seen whatever the window) and with a soft-cap (the sink is not capped)."""
    lens, fps = [300, 129, 40], [0, 500, 77]
    call = _prefill_call(lens, fps, hq=8, hkv=2, window=window, softcap=cap, seed=31, sinks=_sinks(8, 1))
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref)


@pytest.mark.parametrize("window", [0, 1000])
def test_decode_with_sinks(cuda, window):
    """Learned sinks on the split-K decode: the sink joins the merge of the per-chunk partials."""
    call = _decode_call([5000, 1, 2047, 300], hq=8, hkv=2, window=window, seed=32, sinks=_sinks(8, 2))
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_sinks_on_the_generic_path(cuda, kind):
    """fp32 and head_dim 64 go through the CUDA-core kernel; its sinks follow the same definition."""
    if kind == "prefill":
        call = _prefill_call([70, 33], [0, 40], hq=4, hkv=2, d=64, seed=33, sinks=_sinks(4, 3))
    else:
        call = _decode_call([900, 3], hq=4, hkv=2, dtype=torch.float32, seed=34, sinks=_sinks(4, 4))
    ref = ostep.run_layer_call(call)["out"]
    st, _ = _run(call, cuda)
    _close(st.out, ref, fp32=call.dtype == torch.float32)


YARN = {"rope_type": "yarn", "factor": 32.0, "original_max_position_embeddings": 4096, "beta_fast": 32.0,
        "beta_slow": 1.0}


@pytest.mark.parametrize("window,truncate", [(128, False), (0, True)])
def test_yarn_prefill_with_sinks(cuda, window, truncate):
    """A GPT-OSS-style layer (page "Model resolution", gpt_oss: YaRN rotation, a learned sink per head, layers
    alternating a 128-key window and full attention) at positions far past the original context: YaRN's
    ramp and attention factor in the tables, then the tensor-core prefill with sinks."""
    sc = dict(YARN, truncate=truncate)
    call = _prefill_call([100, 37], [9000, 0], hq=8, hkv=2, window=window, seed=41, sinks=_sinks(8, 5),
                         rope_scaling=sc, theta=150000.0, max_pos=131072)
    res = ostep.run_layer_call(call)
    st, _ = _run(call, cuda)
    st.rope()                                   # the tables themselves (the step may fuse them)
    torch.cuda.synchronize()
    n = call.n_tokens
    np.testing.assert_allclose(st.cos[:n].double().cpu().numpy(), res["cos"], atol=5e-7, rtol=0)
    np.testing.assert_allclose(st.sin[:n].double().cpu().numpy(), res["sin"], atol=5e-7, rtol=0)
    _close(st.out, res["out"])


def test_yarn_mscale_ratio_decode(cuda):
    """YaRN with mscale and mscale_all_dim both set (the attention factor is their ratio) on the decode path."""
    sc = dict(YARN, mscale=0.707, mscale_all_dim=0.707 * 1.5)
    call = _decode_call([30000, 5000], hq=8, hkv=2, seed=42, sinks=_sinks(8, 6))
    call.rope_scaling, call.rope_theta, call.max_position_embeddings = sc, 150000.0, 131072
    res = ostep.run_layer_call(call)
    st, _ = _run(call, cuda)
    st.rope()
    torch.cuda.synchronize()
    np.testing.assert_allclose(st.cos[:2].double().cpu().numpy(), res["cos"], atol=5e-7, rtol=0)
    _close(st.out, res["out"])


# (hq, hkv, rotated features): rounds per token = ceil((hq + hkv) / 2); rounds mod 8 = 2, 3, 5, 6, 7, 1, 0, 4
@pytest.mark.parametrize("hq,hkv,rot", [(2, 1, 128), (4, 2, 64), (8, 1, 128), (10, 2, 128), (12, 2, 64),
                                        (16, 2, 128), (24, 8, 96), (6, 2, 128)])
def test_fused_rope_update_head_counts(cuda, hq, hkv, rot):
    """The fused update hands each token's cos/sin fill to the warps with one round fewer (thread index rotated
    by the rounds per token mod 8): every rotation, full and partial rotary, and more tokens than resident
    blocks (stages reused) write the same bits as the table build followed by the plain update. 3517 tokens
    exceed 4 stages x 4 resident blocks x 152 SMs, so every block refills its stages and runs both phases of
    its full/done barriers."""
    from decoder_attention_gb300 import _abi as ab_, step
    call = _prefill_call([2900, 617], [0, 40], hq=hq, hkv=hkv, rot=rot, seed=50 + hq)
    props = torch.cuda.get_device_properties(cuda)
    assert call.n_tokens > 4 * 4 * props.multi_processor_count
    a, b = call.to(cuda), call.to(cuda)
    sa, sb = step.AttentionStep(a, fused_rope=True), step.AttentionStep(b, fused_rope=False)
    assert ab_.kv_rope_fused_supported(sa.L)
    sa.update()
    sb.update()
    torch.cuda.synchronize()
    ab_.check_device_error()
    assert torch.equal(sa.q_rot, sb.q_rot)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


def test_fused_rope_update_many_tokens_per_block(cuda):
    """A fused-update block reads its tokens' rows, positions and lengths 64 tokens ahead into shared memory and
    rereads the next 64 once it has passed them. 47000 tokens over 4 x 152 resident blocks give every block more
    than 64, so each one refills that table; three chunks put LongRoPE's seq_len switch on both sides (30000 and
    15100 above the original 4096, 2000 below). Bits must equal the table build followed by the plain update."""
    from decoder_attention_gb300 import _abi as ab_, inputs, step
    call = _prefill_call([30000, 15000, 2000], [0, 100, 0], hq=2, hkv=1, rot=96, seed=91,
                         rope_scaling=inputs.phi4_longrope_scaling(48), max_pos=131072)
    props = torch.cuda.get_device_properties(cuda)
    assert call.n_tokens > 64 * 4 * props.multi_processor_count
    a, b = call.to(cuda), call.to(cuda)
    sa, sb = step.AttentionStep(a, fused_rope=True), step.AttentionStep(b, fused_rope=False)
    assert ab_.kv_rope_fused_supported(sa.L)
    sa.update()
    sb.update()
    torch.cuda.synchronize()
    ab_.check_device_error()
    assert torch.equal(sa.q_rot, sb.q_rot)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


@pytest.mark.parametrize("number", [2, 3, 4, 5])
def test_fused_rope_update_matches_two_calls(cuda, number):
    """da_kv_cache_update_rope (cos/sin formed in the kernel) writes the same bits as da_rope_tables_build
    followed by da_kv_cache_update: q/k norm, llama3, LongRoPE with its seq_len switch and partial rotary
    (workload 5), contiguous caches and a paged pool."""
    from decoder_attention_gb300 import _abi as ab_, inputs, step
    wl = inputs.make(number, scale="small")
    for call in wl.layers:
        if call.dtype != torch.bfloat16:
            continue
        a, b = call.to(cuda), call.to(cuda)
        sa, sb = step.AttentionStep(a, fused_rope=True), step.AttentionStep(b, fused_rope=False)
        assert ab_.kv_rope_fused_supported(sa.L)
        sa.update()
        sb.update()
        torch.cuda.synchronize()
        ab_.check_device_error()
        assert torch.equal(sa.q_rot, sb.q_rot)
        assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    call = wl.layers[0]
    a, b = call.to(cuda), call.to(cuda)
    kpa, vpa, ta = inputs.paged_from_contiguous(a.k_cache, a.v_cache, 64, seed=5)
    kpb, vpb, tb = inputs.paged_from_contiguous(b.k_cache, b.v_cache, 64, seed=5)
    pa = step.PagedAttentionStep(a, kpa, vpa, ta, 64, fused_rope=True)
    pb = step.PagedAttentionStep(b, kpb, vpb, tb, 64, fused_rope=False)
    pa.update()
    pb.update()
    torch.cuda.synchronize()
    ab_.check_device_error()
    bits = lambda t: t.view(torch.int16)                # the pools hold NaN in spare blocks: compare bits
    assert torch.equal(pa.q_rot, pb.q_rot) and torch.equal(bits(kpa), bits(kpb)) and torch.equal(bits(vpa), bits(vpb))


@pytest.mark.parametrize("hq,window", [(6, 0), (8, 256)])
def test_softcap_both_tanh_forms(cuda, hq, window):
    """Capped prefill tiles take one of two tanh forms per warp: a polynomial when every score of the warp's 32
    rows is small against the cap, else the MUFU tanh. Query rows scaled by 1 and by 12 in alternate blocks of
    32 send alternate warps down each form (cap 5: |scale q.k / cap| stays below 0.3 in the first and reaches
    well past 0.5 in the second); both must match the oracle with its rotated q/k rounded to bf16 as stored."""
    call = _prefill_call([300, 200], [0, 500], hq=hq, hkv=2, window=window, softcap=5.0, seed=70 + hq)
    row = torch.cat([torch.arange(300), torch.arange(200)])
    factor = torch.where((row // 32) % 2 == 0, 1.0, 12.0)
    call.q = (call.q.float() * factor[:, None, None]).to(call.q.dtype)
    st, _ = _run(call, cuda)
    ref = ostep.run_layer_call(call, storage_rounding=True)
    _close(st.out, ref["out"])
    nocap = copy.copy(call)
    nocap.softcap = 0.0
    assert np.abs(ostep.run_layer_call(nocap, storage_rounding=True)["out"] - ref["out"]).max() > 0.1


@pytest.mark.parametrize("window", [0, 256])
def test_cached_decode_equals_recompute(cuda, window):
    """The [MoE/decoding guide] sanity check that cached decoding equals recomputing the whole sequence: token
    T decoded against the cache a prefill of tokens 0..T-1 wrote gives row T of a prefill of tokens 0..T, both
    through the C ABI (the decode and the prefill kernels), and both match the oracle."""
    from decoder_attention_gb300 import inputs, step
    T, hq, hkv = 700, 8, 2
    full = _prefill_call([T + 1], [0], hq=hq, hkv=hkv, window=window, seed=80)
    ref = ostep.run_layer_call(full)["out"]
    st_full = step.AttentionStep(full.to(cuda))
    st_full.run()

    def sub(idx, prefill):
        i = torch.as_tensor(idx)
        n = len(idx)
        qs, tr, tp, tl = inputs._prefill_meta([n], [0], [0]) if prefill else (None, [0], [idx[0]], [idx[0] + 1])
        return inputs.LayerCall(
            head_dim=128, num_attention_heads=hq, num_key_value_heads=hkv, partial_rotary_factor=1.0,
            rope_theta=full.rope_theta, rope_scaling=None, max_position_embeddings=full.max_position_embeddings,
            dtype=full.dtype, window=window, softcap=0.0, q=full.q[i], k=full.k[i], v=full.v[i],
            tok_rows=inputs._i32(tr), tok_pos=inputs._i32(tp), tok_seq_len=inputs._i32(tl),
            n_prefill=n if prefill else 0, q_start=inputs._i32(qs if prefill else [0]),
            pf_rows=inputs._i32([0] if prefill else []), pf_first_pos=inputs._i32([0] if prefill else []),
            max_q_len=n if prefill else 0, dec_rows=inputs._i32([] if prefill else [0]),
            dec_pos=inputs._i32([] if prefill else [idx[0]]), k_cache=full.k_cache, v_cache=full.v_cache)

    pre = sub(list(range(T)), True).to(cuda)
    dec = sub([T], False)
    dec.k_cache, dec.v_cache = pre.k_cache, pre.v_cache          # the cache the prefill writes
    dec = step.AttentionStep(dec.to(cuda))
    step.AttentionStep(pre).run()
    dec.run()
    torch.cuda.synchronize()
    _abi().check_device_error()
    got_dec = dec.out[0].double().cpu().numpy()
    got_full = st_full.out[T].double().cpu().numpy()
    _close(dec.out[0:1], ref[T:T + 1])
    _close(st_full.out[T:T + 1], ref[T:T + 1])
    assert np.abs(got_dec - got_full).max() <= BF16_MAX
