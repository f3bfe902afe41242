"""Plain fp64 CPU oracle for the projections on either side of the attention step (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may import it; the CUDA
library never calls it and shares no code with it.

Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", DecoderAttention:
q = q_proj(x), k = k_proj(x), v = v_proj(x) (nn.Linear, with a bias when qkv_bias), viewed as heads, then the
norms, RoPE and cache.update; after attention, o_proj (with a bias when o_bias) maps the concatenated heads
back to hidden_size. Reading P1: the fused projection's weight stacks the rows of q_proj, k_proj and v_proj in
that order ([(Hq + 2 Hkv) d, hidden]), its bias likewise.
"""
from __future__ import annotations

import numpy as np

from . import attention as A

F64 = np.float64


def qkv_project(x, w_qkv, hq, hkv, d, bias=None):
    """x [N, hidden] -> q [N, hq, d], k [N, hkv, d], v [N, hkv, d]: y = x W^T (+ b), split by rows of W (P1)."""
    y = np.asarray(x, dtype=F64) @ np.asarray(w_qkv, dtype=F64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=F64)
    n = y.shape[0]
    q = y[:, :hq * d].reshape(n, hq, d)
    k = y[:, hq * d:(hq + hkv) * d].reshape(n, hkv, d)
    v = y[:, (hq + hkv) * d:].reshape(n, hkv, d)
    return q, k, v


def project_and_update(layer: A.Layer, x, w_qkv, rows, positions, cos, sin, k_cache, v_cache, bias=None):
    """The projection followed by the step's norm, RoPE and cache write; returns q_rot (caches updated)."""
    q, k, v = qkv_project(x, w_qkv, layer.num_attention_heads, layer.num_key_value_heads, layer.head_dim, bias)
    return A.kv_cache_update(layer, q, k, v, rows, positions, cos, sin, k_cache, v_cache)


def o_project(attn, w_o, bias=None):
    """attn [N, hq, d] -> [N, hidden]: the heads concatenated, times W_o^T (+ b)."""
    a = np.asarray(attn, dtype=F64)
    y = a.reshape(a.shape[0], -1) @ np.asarray(w_o, dtype=F64).T
    if bias is not None:
        y = y + np.asarray(bias, dtype=F64)
    return y
