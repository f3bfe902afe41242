"""Full-size workloads through the same calls bench.py times, checked on sampled outputs.

Each workload runs whole on the GPU; the oracle then recomputes a sample of the outputs one query at a time.
Its inputs are the workload's own: the new tokens' q/k/v (rotated by the oracle itself) and, for keys that
were already cached, the cache rows copied to the host before any kernel ran. Tolerances are the bf16 ones
of the parity tests (max-abs 2e-2, mean-abs 2e-3 over the sampled outputs).
"""
import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import step as ostep

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 2e-3


def _np64(t):
    return t.detach().to("cpu").double().numpy()


def _check(diffs):
    d = np.concatenate([x.ravel() for x in diffs])
    assert np.isfinite(d).all()
    assert d.max() <= BF16_MAX and d.mean() <= BF16_MEAN, (d.max(), d.mean())


def _prefill_samples(call, st, snap, rng, n_samples=24):
    """Sampled (token, head) outputs of the prefill chunks. snap: {row: (K, V)} host copies of the rows
    before the step (keys before each chunk's first position come from there)."""
    layer = ostep.layer_of(call)
    qs = call.q_start.cpu().numpy()
    fps = call.pf_first_pos.cpu().numpy()
    rows = call.pf_rows.cpu().numpy()
    out = st.out
    diffs = []
    for _ in range(n_samples):
        b = int(rng.integers(len(rows)))
        if int(rows[b]) not in snap:
            continue
        n_b = int(qs[b + 1] - qs[b])
        i = int(rng.integers(n_b))
        p = int(fps[b]) + i
        toks = np.arange(qs[b], qs[b] + i + 1)                 # the chunk's tokens up to the query
        q_rot, k_rot = ostep.rotate_tokens(call, toks)
        K0, V0 = snap[int(rows[b])]
        lo = max(0, p - call.window + 1) if call.window else 0
        kk = np.concatenate([_np64(K0[:, lo:int(fps[b])]), k_rot.transpose(1, 0, 2)[:, max(0, lo - int(fps[b])):]],
                            axis=1)
        vv = np.concatenate([_np64(V0[:, lo:int(fps[b])]),
                             _np64(call.v[toks]).transpose(1, 0, 2)[:, max(0, lo - int(fps[b])):]], axis=1)
        kp = np.arange(lo, p + 1)
        ref = A.causal_attention(q_rot[-1:], kk, vv, [p], kp, call.window, call.softcap, 0.0)[0]
        h = int(rng.integers(call.num_attention_heads))
        got = out[int(qs[b]) + i, h].double().cpu().numpy()
        diffs.append(np.abs(got - ref[h]))
    return diffs


def _decode_samples(call, st, snap, which):
    """Sampled decode outputs; snap[row] = (K, V) host bf16 copies of slots [lo, p) of the row, lo the first
    visible key of the row's query."""
    npf = call.n_prefill
    pos = call.dec_pos.cpu().numpy()
    rows = call.dec_rows.cpu().numpy()
    diffs = []
    for s in which:
        p, row = int(pos[s]), int(rows[s])
        lo = max(0, p - call.window + 1) if call.window else 0
        q_rot, k_rot = ostep.rotate_tokens(call, [npf + s])
        K0, V0 = snap[(row, lo)]
        K = np.concatenate([_np64(K0), k_rot[0][:, None, :]], axis=1)
        V = np.concatenate([_np64(V0), _np64(call.v[npf + s])[:, None, :]], axis=1)
        ref = A.causal_attention(q_rot, K, V, [p], np.arange(lo, p + 1), call.window, call.softcap, 0.0)[0]
        got = st.out[npf + s].double().cpu().numpy()
        diffs.append(np.abs(got - ref))
    return diffs


def _snap_decode(call, which):
    pos = call.dec_pos.cpu().numpy()
    rows = call.dec_rows.cpu().numpy()
    out = {}
    for s in which:
        p, row = int(pos[s]), int(rows[s])
        lo = max(0, p - call.window + 1) if call.window else 0
        out[(row, lo)] = (call.k_cache[row, :, lo:p].cpu(), call.v_cache[row, :, lo:p].cpu())
    return out


def _run(wl):
    from decoder_attention_gb300 import _abi, step
    steps = [step.AttentionStep(c) for c in wl.layers]
    for s in steps:
        s.run()
    torch.cuda.synchronize()
    _abi.check_device_error()
    return steps


def _snap(call, rows, upto):
    """Host copies (cache dtype) of cache rows, slots [0, upto)."""
    return {int(r): (call.k_cache[int(r), :, :upto].cpu(), call.v_cache[int(r), :, :upto].cpu()) for r in rows}


def test_qwen3_8b_prefill_full(cuda):
    from decoder_attention_gb300 import inputs
    wl = inputs.make(2, scale="full", device=cuda)
    call = wl.layers[0]
    snap = _snap(call, range(call.num_rows), 1)          # the chunks start at position 0: nothing cached
    st = _run(wl)[0]
    _check(_prefill_samples(call, st, snap, np.random.default_rng(0), 32))


@pytest.mark.parametrize("number", [3, 4])
def test_decode_full(cuda, number):
    from decoder_attention_gb300 import inputs
    wl = inputs.make(number, scale="full", device=cuda)
    call = wl.layers[0]
    S = call.n_decode
    which = sorted(set([0, S - 1] + list(np.random.default_rng(number).integers(0, S, 2 if number == 3 else 0))))
    snap = _snap_decode(call, which)
    st = _run(wl)[0]
    _check(_decode_samples(call, st, snap, which))


def test_phi4_gemma2_mixed_full(cuda):
    from decoder_attention_gb300 import inputs
    wl = inputs.make(5, scale="full", device=cuda)
    rng = np.random.default_rng(5)
    snaps = []
    for call in wl.layers:
        pf_rows = call.pf_rows.cpu().numpy()[:1]
        dec_idx = [0, 1, call.n_decode - 1]
        upto = int(call.pf_first_pos.max()) + 1
        snaps.append((_snap(call, pf_rows, upto), _snap_decode(call, dec_idx), dec_idx))
    steps = _run(wl)
    diffs = []
    for call, st, (psnap, dsnap, dec_idx) in zip(wl.layers, steps, snaps):
        diffs += _prefill_samples(call, st, psnap, rng, 12)
        diffs += _decode_samples(call, st, dsnap, dec_idx)
    _check(diffs)


def test_qwen3_8b_prefill_whole_sequence(cuda):
    """One whole chunk of the Qwen3-8B-shaped prefill, every query and every head (2048 x 32 outputs),
    element by element against the oracle on the chunk's own rotated keys (the chunks start at position 0)."""
    from decoder_attention_gb300 import inputs
    wl = inputs.make(2, scale="full", device=cuda)
    call = wl.layers[0]
    st = _run(wl)[0]
    qs = call.q_start.cpu().numpy()
    b = 2                                                 # a chunk in the middle of the batch
    toks = np.arange(qs[b], qs[b + 1])
    q_rot, k_rot = ostep.rotate_tokens(call, toks)
    pos = np.arange(len(toks))
    ref = A.causal_attention(q_rot, k_rot.transpose(1, 0, 2), _np64(call.v[toks]).transpose(1, 0, 2), pos, pos,
                             call.window, call.softcap, 0.0)
    got = st.out[int(qs[b]):int(qs[b + 1])].double().cpu().numpy()
    _check([np.abs(got - ref)])


def test_llama31_decode_every_sequence_one_kv_group(cuda):
    """Every sequence of the Llama-3.1-8B-shaped decode (16 x 131072 keys, split-K over many chunks) for the
    query heads of KV head 0, against the oracle on the cache rows copied before the step."""
    from decoder_attention_gb300 import inputs
    wl = inputs.make(4, scale="full", device=cuda)
    call = wl.layers[0]
    G = call.num_attention_heads // call.num_key_value_heads
    pos = call.dec_pos.cpu().numpy()
    rows = call.dec_rows.cpu().numpy()
    snap = [(call.k_cache[int(r), 0:1, :int(p)].cpu(), call.v_cache[int(r), 0:1, :int(p)].cpu()) for r, p in zip(rows, pos)]
    st = _run(wl)[0]
    npf = call.n_prefill
    diffs = []
    for s in range(call.n_decode):
        p = int(pos[s])
        q_rot, k_rot = ostep.rotate_tokens(call, [npf + s])
        K = np.concatenate([_np64(snap[s][0]), k_rot[0][0:1, None, :]], axis=1)
        V = np.concatenate([_np64(snap[s][1]), _np64(call.v[npf + s])[0:1, None, :]], axis=1)
        ref = A.causal_attention(q_rot[:, :G], K, V, [p], np.arange(p + 1), call.window, call.softcap, 0.0)[0]
        diffs.append(np.abs(st.out[npf + s, :G].double().cpu().numpy() - ref))
    _check(diffs)
