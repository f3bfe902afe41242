"""Host-side pieces of bench.py's CPU baselines (no GPU): the bounded samples it hands the oracle.

The all-cores baseline cuts its sample into (chunk or token, KV-head group) units; attention of different KV-head
groups is independent (each query head reads its own group's keys), so the units' outputs, put back together,
must equal the oracle's output on the whole sample, and their work must add up to the whole sample's.
"""
import numpy as np
import torch

from oracle import step as ostep


def test_kv_head_units_reassemble_the_whole_call():
    from decoder_attention_gb300 import inputs, work as W
    call = inputs.make(5, scale="small").layers[1]          # prefill chunks and decode tokens, Hq 6, Hkv 2
    whole = inputs.subset(call, [0, 1], [0, 2])
    ref = ostep.run_layer_call(whole)["out"]
    G = call.num_attention_heads // call.num_key_value_heads
    parts = [inputs.subset(call, [0, 1], [0, 2], kv_heads=1, kv_first=g) for g in range(call.num_key_value_heads)]
    outs = [ostep.run_layer_call(p)["out"] for p in parts]
    np.testing.assert_array_equal(np.concatenate(outs, axis=1), ref)
    for g, p in enumerate(parts):
        assert p.num_attention_heads == G and p.num_key_value_heads == 1
        assert torch.equal(p.q, whole.q[:, g * G:(g + 1) * G])
    tot = {}
    for p in parts:
        for k, v in W.layer_call_work(p).items():
            tot[k] = tot.get(k, 0) + v
    w = W.layer_call_work(whole)
    for k in ("prefill_flops", "decode_bytes", "decode_flops", "prefill_pairs"):
        assert tot[k] == w[k], k


def test_headline_units():
    import bench
    v, u, tps = bench.headline({"prefill_flops": 2e12, "decode_flops": 0, "decode_bytes": 0, "tokens": 100}, 2.0)
    assert (v, u, tps) == (1.0, "TFLOP/s", 50.0)
    v, u, tps = bench.headline({"prefill_flops": 0, "decode_flops": 1, "decode_bytes": 4e9, "tokens": 8}, 2.0)
    assert (v, u, tps) == (2.0, "GB/s", 4.0)
