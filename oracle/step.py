"""Run the fp64 oracle on one layer call of the synthetic workloads (TEST INFRASTRUCTURE ONLY).

The call object is read by attribute (q, k, v, tok_rows, ... as the workload generator lays them out);
nothing of the CUDA library is imported or called here.
"""
from __future__ import annotations

import numpy as np

from . import attention as A


def _np64(t):
    return t.detach().to("cpu").double().numpy()


def _np_int(t):
    return t.detach().to("cpu").numpy().astype(np.int64)


def layer_of(call) -> A.Layer:
    rot = A.rotary_dim(call.head_dim, call.partial_rotary_factor)
    return A.Layer(head_dim=call.head_dim, num_attention_heads=call.num_attention_heads,
                   num_key_value_heads=call.num_key_value_heads, rotary_dim=rot,
                   q_norm_w=_np64(call.q_norm_w) if call.q_norm_w is not None else None,
                   k_norm_w=_np64(call.k_norm_w) if call.k_norm_w is not None else None,
                   eps=call.eps, window=call.window, softcap=call.softcap, scale=0.0,
                   sinks=_np64(call.sinks) if getattr(call, "sinks", None) is not None else None)


def spec_of(call) -> A.RopeSpec:
    return A.RopeSpec(theta=call.rope_theta, scaling=call.rope_scaling,
                      max_position_embeddings=call.max_position_embeddings)


def rope_tables(call, positions=None, seq_len=None):
    layer = layer_of(call)
    pos = _np_int(call.tok_pos) if positions is None else np.asarray(positions)
    lens = _np_int(call.tok_seq_len) if seq_len is None else np.asarray(seq_len)
    return A.rope_tables_for_tokens(spec_of(call), layer.rotary_dim, pos, lens)


def round_to_storage(x, dtype):
    """x rounded once to the storage type `dtype` (torch dtype; round to nearest even), back in float64.

    The pages' engine keeps rotated queries and cached keys in the activation dtype (page "42. More models",
    section "Scaled RoPE": rope_tables casts cos/sin to that dtype, and the cache holds that dtype); a bf16
    cache therefore carries each rotated key rounded to bf16. Oracle values only pass through here."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).double().numpy()


def run_layer_call(call, key_positions=None, storage_rounding=False):
    """All results of one call at a size the oracle handles whole: cos, sin, q_rot, caches after the
    update, and the attention output of every token (float64). With storage_rounding, the oracle's own
    rotated q and k are rounded to the call's dtype before attention, as a cache of that dtype stores them."""
    layer = layer_of(call)
    cos, sin = rope_tables(call)
    kc = _np64(call.k_cache).copy()
    vc = _np64(call.v_cache).copy()
    rows, pos = _np_int(call.tok_rows), _np_int(call.tok_pos)
    q_rot = A.kv_cache_update(layer, _np64(call.q), _np64(call.k), _np64(call.v), rows, pos, cos, sin, kc, vc)
    if storage_rounding:
        q_rot = round_to_storage(q_rot, call.dtype)
        for t in range(len(rows)):
            kc[rows[t], :, pos[t]] = round_to_storage(kc[rows[t], :, pos[t]], call.dtype)
    out = np.zeros_like(q_rot)
    npf = call.n_prefill
    kp = None if key_positions is None else _np_int(key_positions)
    if npf:
        out[:npf] = A.attn_prefill(layer, q_rot[:npf], kc, vc, _np_int(call.q_start), _np_int(call.pf_rows),
                                   _np_int(call.pf_first_pos), key_positions=kp)
    if call.n_tokens > npf:
        out[npf:] = A.attn_decode(layer, q_rot[npf:], kc, vc, _np_int(call.dec_rows), _np_int(call.dec_pos),
                                  key_positions=kp)
    return {"cos": cos, "sin": sin, "q_rot": q_rot, "k_cache": kc, "v_cache": vc, "out": out}


def rotate_tokens(call, token_ids):
    """q_rot [n, Hq, d] and k_rot [n, Hkv, d] of the given tokens of the call (norm + RoPE), float64."""
    layer = layer_of(call)
    idx = np.asarray(token_ids, dtype=np.int64)
    pos = _np_int(call.tok_pos)[idx]
    lens = _np_int(call.tok_seq_len)[idx]
    cos, sin = A.rope_tables_for_tokens(spec_of(call), layer.rotary_dim, pos, lens)
    q = _np64(call.q[idx])
    k = _np64(call.k[idx])
    if layer.q_norm_w is not None:
        q = A.rms_norm(q, layer.q_norm_w, layer.eps)
        k = A.rms_norm(k, layer.k_norm_w, layer.eps)
    c, s = cos[:, None, :], sin[:, None, :]
    return A.apply_rope(q, c, s), A.apply_rope(k, c, s)


def run_layer_call_paged(call, k_pool, v_pool, block_table, block_size):
    """run_layer_call over a paged pool (k_pool/v_pool [n_blocks, Hkv, block_size, d], block_table [R,
    max_blocks]): the cache update writes through the table, and attention reads through it."""
    layer = layer_of(call)
    cos, sin = rope_tables(call)
    kp = _np64(k_pool).copy()
    vp = _np64(v_pool).copy()
    table = _np_int(block_table)
    rows, pos = _np_int(call.tok_rows), _np_int(call.tok_pos)
    q_rot = A.kv_cache_update_paged(layer, _np64(call.q), _np64(call.k), _np64(call.v), rows, pos, cos, sin, kp, vp,
                                    table, block_size)
    out = np.zeros_like(q_rot)
    npf = call.n_prefill
    if npf:
        out[:npf] = A.attn_prefill_paged(layer, q_rot[:npf], kp, vp, table, block_size, _np_int(call.q_start),
                                         _np_int(call.pf_rows), _np_int(call.pf_first_pos))
    if call.n_tokens > npf:
        out[npf:] = A.attn_decode_paged(layer, q_rot[npf:], kp, vp, table, block_size, _np_int(call.dec_rows),
                                        _np_int(call.dec_pos))
    return {"cos": cos, "sin": sin, "q_rot": q_rot, "k_pool": kp, "v_pool": vp, "out": out}
