"""Plain fp64 CPU oracle for multi-head latent attention decode with absorbed up-projections.

THIS MODULE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import it. The CUDA library never calls it and shares no code with it.

It restates the page "42. More models: a registry, scaled RoPE, sliding windows and latent attention"
(inference.shantanugoel.com), section "Multi-head latent attention" and its subsection "Serving it: absorbing
the up-projections": each token caches one row [c, k_rope] (the latent c of width kv_lora_rank, then its
rotary key of width qk_rope_head_dim), every query head maps its non-rotary part into latent space once
(q_latent = W_uk^T q_nope), and attention is multi-query attention of all heads against the cached rows,
whose first kv_lora_rank features are the values; W_uv maps each head's latent output back afterwards.

Readings where the page leaves a step open:

  M1  rotary features of DeepSeek checkpoints pair adjacent elements (0, 1), (2, 3), ...; they are
      deinterleaved (even elements, then odd ones) and rotated by the split-half rotation, for queries and
      keys alike, and the cache holds the deinterleaved, rotated k_rope.
  M2  the softmax scale is (qk_nope_head_dim + qk_rope_head_dim)^-0.5, times (0.1 mscale_all_dim ln s + 1)^2
      when rope_scaling has mscale_all_dim and a factor s > 1 (YaRN's temperature on the scale).
  M3  a decode token at position p of cache row r sees rows 0..p of that cache row (slot = position).
"""
from __future__ import annotations

import math

import numpy as np

from .attention import apply_rope

F64 = np.float64


def deinterleave(x):
    """Adjacent pairs (0, 1), (2, 3), ... reordered to split-half pairs (i, i + r/2): evens, then odds (M1)."""
    x = np.asarray(x, dtype=F64)
    return np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)


def mla_scale(qk_nope_head_dim, qk_rope_head_dim, rope_scaling=None):
    """Softmax scale of MLAAttention (M2)."""
    scale = (qk_nope_head_dim + qk_rope_head_dim) ** -0.5
    s = rope_scaling or {}
    if s.get("mscale_all_dim") and s.get("factor", 1.0) > 1:
        m = 0.1 * s["mscale_all_dim"] * math.log(s["factor"]) + 1.0
        scale *= m * m
    return scale


def mla_rope(x, cos, sin):
    """Deinterleave then split-half rotate the rotary features x [N, ..., r] with cos/sin [N, r/2] (M1)."""
    x = deinterleave(x)
    c = np.asarray(cos, dtype=F64)
    s = np.asarray(sin, dtype=F64)
    while c.ndim < x.ndim:
        c, s = c[:, None], s[:, None]
    return apply_rope(x, c, s)


def mla_cache_update(latent, k_rope, rows, positions, cos, sin, cache):
    """Writes row [c, rotated k_rope] of token t at cache[rows[t], positions[t]] (cache [R, M, rank + r])."""
    latent = np.asarray(latent, dtype=F64)
    kr = mla_rope(k_rope, cos, sin)
    for t in range(latent.shape[0]):
        cache[rows[t], positions[t]] = np.concatenate([latent[t], kr[t]])


def mla_query(q_latent, q_rope, cos, sin):
    """The absorbed query of each head, [N, H, rank + r]: [W_uk^T q_nope, rotated q_rope] (M1)."""
    return np.concatenate([np.asarray(q_latent, dtype=F64), mla_rope(q_rope, cos, sin)], axis=-1)


def mla_decode(q, cache, rows, positions, scale, rank, window=0):
    """Absorbed MLA decode: q [S, H, rank + r] against cache rows [R, M, rank + r]; token s at position p of
    row rows[s] sees rows 0..p (M3; with a window w, p - w + 1 .. p). Returns the latent outputs [S, H, rank]:
    out[s, h] = sum_j softmax_j(scale * q[s, h] . row_j) row_j[:rank]."""
    q = np.asarray(q, dtype=F64)
    S, H, _ = q.shape
    out = np.zeros((S, H, rank), dtype=F64)
    for s in range(S):
        p, r = int(positions[s]), int(rows[s])
        lo = max(0, p - window + 1) if window else 0
        kv = np.asarray(cache[r, lo:p + 1], dtype=F64)            # [n, rank + r]
        z = scale * (q[s] @ kv.T)                                  # [H, n]
        z = z - z.max(axis=1, keepdims=True)
        e = np.exp(z)
        w = e / e.sum(axis=1, keepdims=True)
        out[s] = w @ kv[:, :rank]
    return out


def run_mla_call(call):
    """The oracle over one MLA decode step (the call object of the workload generator, read by attribute):
    tables for the rotary features, the cache update, the absorbed queries and the decode (float64)."""
    from .attention import rope_inv_freq, rope_tables
    pos = call.positions.detach().cpu().numpy().astype(np.int64)
    rows = call.rows.detach().cpu().numpy().astype(np.int64)
    inv, af = rope_inv_freq(call.qk_rope_head_dim, call.rope_theta, call.rope_scaling, call.max_position_embeddings)
    cos, sin = rope_tables(pos, inv, af)
    cache = call.cache.detach().cpu().double().numpy().copy()
    q = call.q.detach().cpu().double().numpy()
    mla_cache_update(call.latent.detach().cpu().double().numpy(), call.k_rope.detach().cpu().double().numpy(), rows,
                     pos, cos, sin, cache)
    rank = q.shape[-1] - call.qk_rope_head_dim
    q_rot = mla_query(q[..., :rank], q[..., rank:], cos, sin)
    scale = mla_scale(call.qk_nope_head_dim, call.qk_rope_head_dim, call.rope_scaling)
    out = mla_decode(q_rot, cache, rows, pos, scale, rank, call.window)
    return {"cos": cos, "sin": sin, "cache": cache, "q_rot": q_rot, "out": out}
