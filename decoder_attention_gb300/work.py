"""Algorithmic work of one attention step, counted over allowed (query, key) pairs only.

Prefill: FLOPs = 4 * d * sum over queries and query heads of the visible keys (2 for q.k, 2 for p.v per
key and dim); one exp per visible pair. Decode: bytes = visible keys * 2 (K and V) * Hkv * d * element
size, each cached key read once per KV head group. Masked lanes of boundary tiles and skipped tiles
count for nothing. Page "42. More models: ...", section "Multi-head latent attention" prints the per-token
KV cache sizes (e.g. 128 KiB for Llama-3.1-8B's 32 layers) that the same per-key figure reproduces.
"""
from __future__ import annotations

import torch


def visible_keys(position: int, window: int) -> int:
    """Keys a query at `position` sees: itself and the earlier ones, at most `window` (0 = no window)."""
    n = position + 1
    return min(n, window) if window else n


def kv_bytes_per_key(hkv: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K and V bytes of one cached key of one layer."""
    return 2 * hkv * head_dim * elem_bytes


def _visible_sum(p0: int, n: int, window: int) -> int:
    """sum_{i < n} visible_keys(p0 + i, window), in closed form."""
    if n <= 0:
        return 0
    if not window:
        a, b = p0 + 1, p0 + n
        return (a + b) * n // 2
    # positions with p + 1 <= window see p + 1 keys, the rest see `window`
    first_full = max(p0, window - 1)            # first position that sees exactly `window` keys
    n_grow = max(0, min(n, first_full - p0))    # positions p0 .. first_full - 1
    a, b = p0 + 1, p0 + n_grow
    return (a + b) * n_grow // 2 + (n - n_grow) * window


def layer_call_work(call) -> dict:
    """FLOPs, exps, KV bytes and token counts of one LayerCall (workload generator layout)."""
    hq, hkv, d = call.num_attention_heads, call.num_key_value_heads, call.head_dim
    elem = 4 if call.dtype == torch.float32 else 2
    qs = call.q_start.cpu().tolist()
    fps = call.pf_first_pos.cpu().tolist()
    pairs_pf = 0
    for b in range(len(fps)):
        pairs_pf += _visible_sum(int(fps[b]), int(qs[b + 1] - qs[b]), call.window)
    keys_dec = sum(visible_keys(int(p), call.window) for p in call.dec_pos.cpu().tolist())
    # prefill reads each (row, KV head) key range once per query tile in principle; its algorithmic bytes
    # are Q + K + V + O once
    pf_bytes = 0
    if call.n_prefill:
        kv_keys = sum(int(fps[b]) + int(qs[b + 1] - qs[b]) for b in range(len(fps)))
        pf_bytes = call.n_prefill * hq * d * elem * 2 + kv_keys * kv_bytes_per_key(hkv, d, elem)
    return {
        "prefill_pairs": pairs_pf * hq,
        "prefill_flops": 4 * d * pairs_pf * hq,
        "prefill_exps": pairs_pf * hq,
        "prefill_bytes": pf_bytes,
        "decode_keys": keys_dec,
        "decode_bytes": keys_dec * kv_bytes_per_key(hkv, d, elem),
        "decode_flops": 4 * d * keys_dec * hq,
        "tokens": call.n_tokens,
        "prefill_tokens": call.n_prefill,
        "decode_tokens": call.n_decode,
    }


def workload_work(workload) -> dict:
    tot = {}
    for call in workload.layers:
        for k, v in layer_call_work(call).items():
            tot[k] = tot.get(k, 0) + v
    return tot
