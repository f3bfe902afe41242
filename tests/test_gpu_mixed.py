"""da_attn_mixed on the GPU: a mixed batch's prefill chunks and decode tokens in one call, the two run side by
side when the split model says it pays. Every output must be bit for bit what da_attn_prefill followed by
da_attn_decode writes (the same kernels compute each output; only the SMs they share differ), on contiguous
caches and a paged pool, on a non-default stream whose next operation must see both parts, and inside a CUDA
graph capture. The oracle check of the mixed layer pair at full size runs through the same call
(`AttentionStep.run`, in test_gpu_fullsize.py)."""
import numpy as np
import pytest
import torch

from oracle import step as ostep

pytestmark = pytest.mark.gpu

# Hints shaped like the mixed layer pair's full layer (8 chunks x 1024 tokens at ~33K context, 120 decode
# tokens at ~33K): the split model then gives the prefill part of the SMs, whatever the data's real size.
OVERLAP_PAIRS, OVERLAP_KEYS = 8 * 1024 * 33000.0, 120 * 33000.0


def _sequential(st, stream=None):
    st.prefill(stream)
    st.decode(stream)


def _forced_mixed(st, stream=None, paged=False):
    from decoder_attention_gb300 import _abi
    c = st.call
    if paged:
        _abi.attn_mixed_paged(st.L, st.q_rot, st.kv, c.n_prefill, len(c.pf_rows), c.q_start, c.pf_rows,
                              c.pf_first_pos, c.max_q_len, c.n_decode, c.dec_rows, c.dec_pos, OVERLAP_PAIRS,
                              OVERLAP_KEYS, st.out, st.workspace, st.ws_bytes, stream)
    else:
        _abi.attn_mixed(st.L, st.q_rot, c.k_cache, c.v_cache, c.num_rows, c.max_len, c.n_prefill, len(c.pf_rows),
                        c.q_start, c.pf_rows, c.pf_first_pos, c.max_q_len, c.n_decode, c.dec_rows, c.dec_pos,
                        OVERLAP_PAIRS, OVERLAP_KEYS, st.out, st.workspace, st.ws_bytes, stream)


def _mixed_layers(scale="small"):
    from decoder_attention_gb300 import inputs
    return inputs.make(5, scale=scale).layers


def test_split_overlaps_for_the_forced_hints(cuda):
    from decoder_attention_gb300 import _abi, step
    n_sm = torch.cuda.get_device_properties(cuda).multi_processor_count
    for call in _mixed_layers():
        st = step.AttentionStep(call.to(cuda))
        p = _abi.attn_mixed_prefill_sms(st.L, n_sm, OVERLAP_PAIRS, OVERLAP_KEYS)
        assert n_sm // 4 <= p < n_sm, p


@pytest.mark.parametrize("forced", [False, True])
def test_mixed_equals_two_calls(cuda, forced):
    """Workload 5 at its small size (both layers: windowed and full, soft-cap, LongRoPE, partial rotary): with
    the call's own hints (which may choose to run the parts in turn) and with hints that force the overlap."""
    from decoder_attention_gb300 import _abi, step
    for call in _mixed_layers():
        a, b = call.to(cuda), call.to(cuda)
        sa, sb = step.AttentionStep(a), step.AttentionStep(b)
        sa.update()
        sb.update()
        if forced:
            _forced_mixed(sa)
        else:
            sa.attend()
        _sequential(sb)
        torch.cuda.synchronize()
        _abi.check_device_error()
        assert torch.equal(sa.out, sb.out)
        assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)


def test_mixed_paged_equals_two_calls(cuda):
    from decoder_attention_gb300 import _abi, inputs, step
    for call in _mixed_layers():
        a, b = call.to(cuda), call.to(cuda)
        kpa, vpa, ta = inputs.paged_from_contiguous(a.k_cache, a.v_cache, 64, seed=9)
        kpb, vpb, tb = inputs.paged_from_contiguous(b.k_cache, b.v_cache, 64, seed=9)
        pa = step.PagedAttentionStep(a, kpa, vpa, ta, 64)
        pb = step.PagedAttentionStep(b, kpb, vpb, tb, 64)
        pa.update()
        pb.update()
        _forced_mixed(pa, paged=True)
        _sequential(pb)
        torch.cuda.synchronize()
        _abi.check_device_error()
        assert torch.equal(pa.out, pb.out)


def test_mixed_on_a_side_stream_joins_before_the_next_operation(cuda):
    """On a non-default stream, an operation enqueued right after the call (a copy of the output) must see
    both parts: the call joins its own stream back before returning."""
    from decoder_attention_gb300 import _abi, step
    call = _mixed_layers()[1]
    a, b = call.to(cuda), call.to(cuda)
    sa, sb = step.AttentionStep(a), step.AttentionStep(b)
    s = torch.cuda.Stream()
    snap = torch.empty_like(sa.out)
    with torch.cuda.stream(s):
        sa.update(s)
        sa.out.fill_(float("nan"))
        _forced_mixed(sa, s)
        snap.copy_(sa.out)
    sb.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    assert torch.equal(snap, sb.out)


def test_mixed_under_graph_capture(cuda):
    """The fork onto the library's stream and the join back are capturable: a CUDA graph of the step replays to
    the same bits."""
    from decoder_attention_gb300 import _abi, step
    call = _mixed_layers()[0]
    a, b = call.to(cuda), call.to(cuda)
    sa, sb = step.AttentionStep(a), step.AttentionStep(b)
    sa.update()
    _forced_mixed(sa)           # first call outside the capture: the library creates its stream and events
    torch.cuda.synchronize()
    sa.out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _forced_mixed(sa)
    g.replay()
    sb.update()
    _sequential(sb)
    torch.cuda.synchronize()
    _abi.check_device_error()
    assert torch.equal(sa.out, sb.out)


def test_mixed_matches_the_oracle(cuda):
    """The forced-overlap call against the fp64 oracle on workload 5's small size."""
    from decoder_attention_gb300 import _abi, step
    for call in _mixed_layers():
        st = step.AttentionStep(call.to(cuda))
        st.update()
        _forced_mixed(st)
        torch.cuda.synchronize()
        _abi.check_device_error()
        ref = ostep.run_layer_call(call)
        d = np.abs(st.out.double().cpu().numpy() - ref["out"])
        assert np.isfinite(d).all()
        assert d.max() <= 2e-2 and d.mean() <= 2e-3, (d.max(), d.mean())


def test_mixed_from_two_host_threads(cuda):
    """Two host threads, each with its own stream and layer call, enqueue mixed calls at once: the library's
    one fork stream per device and its shared events are used under a lock, so every call still joins its own
    stream after its own two parts (results equal to the two calls made in turn, for every repetition)."""
    import threading
    from decoder_attention_gb300 import _abi, step
    calls = _mixed_layers()
    runs = []
    for call in calls:
        a, b = call.to(cuda), call.to(cuda)
        sa, sb = step.AttentionStep(a), step.AttentionStep(b)
        sa.update()
        sb.update()
        _sequential(sb)
        runs.append((sa, sb))
    torch.cuda.synchronize()
    errors = []

    def worker(sa, sb):
        try:
            torch.cuda.set_device(cuda)
            s = torch.cuda.Stream()
            snaps = []
            with torch.cuda.stream(s):
                for _ in range(8):
                    sa.out.fill_(float("nan"))
                    _forced_mixed(sa, s)
                    snaps.append(sa.out.clone())
            s.synchronize()
            for x in snaps:
                if not torch.equal(x, sb.out):
                    errors.append("mismatch")
        except Exception as e:   # reported to the main thread
            errors.append(repr(e))

    ts = [threading.Thread(target=worker, args=r) for r in runs]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    _abi.check_device_error()
    assert not errors, errors


def test_mixed_with_one_part_or_none(cuda):
    """A mixed call whose batch has only prefill chunks, only decode tokens, or nothing at all runs what there
    is (in turn on the caller's stream) and writes what the separate calls write."""
    from decoder_attention_gb300 import _abi, step
    call = _mixed_layers()[1]
    a, b = call.to(cuda), call.to(cuda)
    sa, sb = step.AttentionStep(a), step.AttentionStep(b)
    sa.update()
    sb.update()
    _sequential(sb)
    torch.cuda.synchronize()
    c = sa.call
    for n_tokens, n_seqs, n_dec in ((c.n_prefill, len(c.pf_rows), 0), (0, 0, c.n_decode), (0, 0, 0)):
        sa.out.fill_(float("nan"))
        # the decode part reads its tokens after the chunks' n_tokens rows: with no chunks, from row 0
        q_rot = sa.q_rot if n_tokens or not n_dec else sa.q_rot[c.n_prefill:]
        out = sa.out if n_tokens or not n_dec else sa.out[c.n_prefill:]
        _abi.attn_mixed(sa.L, q_rot, c.k_cache, c.v_cache, c.num_rows, c.max_len, n_tokens, n_seqs, c.q_start,
                        c.pf_rows, c.pf_first_pos, c.max_q_len, n_dec, c.dec_rows, c.dec_pos, OVERLAP_PAIRS,
                        OVERLAP_KEYS, out, sa.workspace, sa.ws_bytes)
        torch.cuda.synchronize()
        _abi.check_device_error()
        if n_tokens:
            assert torch.equal(sa.out[:c.n_prefill], sb.out[:c.n_prefill])
            assert torch.isnan(sa.out[c.n_prefill:].float()).all()
        elif n_dec:
            assert torch.equal(sa.out[c.n_prefill:], sb.out[c.n_prefill:])
            assert torch.isnan(sa.out[:c.n_prefill].float()).all()
        else:
            assert torch.isnan(sa.out.float()).all()
