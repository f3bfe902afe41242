"""ctypes binding of libdecattn.so (include/decattn.h): argument marshalling only.

Every function here takes torch tensors for device memory, passes their data pointers, sizes and the
current CUDA stream to the C entry point of the same name (without the ``da_`` prefix), and raises
``DecAttnError`` with the library's message when the call returns nonzero. No arithmetic of the step
happens in Python: if the library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdecattn.so")

DA_OK = 0
DA_ERR_INVALID_ARG = -1
DA_ERR_UNSUPPORTED = -2
DA_ERR_CUDA = -3
DA_ERR_DEVICE_INDEX = -4
DA_ERR_TIMEOUT = -5
DA_ERR_OUT_OF_BLOCKS = -6

DA_ROPE_DEFAULT, DA_ROPE_LINEAR, DA_ROPE_LLAMA3, DA_ROPE_LONGROPE, DA_ROPE_YARN = range(5)
DA_BF16, DA_FP32 = 0, 1
ROPE_KINDS = {"default": DA_ROPE_DEFAULT, "linear": DA_ROPE_LINEAR, "llama3": DA_ROPE_LLAMA3,
              "longrope": DA_ROPE_LONGROPE, "yarn": DA_ROPE_YARN}
DTYPES = {torch.bfloat16: DA_BF16, torch.float32: DA_FP32}


class DecAttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"decattn error {code}: {msg}")
        self.code = code


class DaRopeScaling(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("theta", ctypes.c_double), ("rotary_dim", ctypes.c_int),
                ("factor", ctypes.c_double), ("low_freq_factor", ctypes.c_double),
                ("high_freq_factor", ctypes.c_double), ("original_max_position_embeddings", ctypes.c_int),
                ("max_position_embeddings", ctypes.c_int), ("short_factor", ctypes.POINTER(ctypes.c_double)),
                ("long_factor", ctypes.POINTER(ctypes.c_double)), ("attention_factor", ctypes.c_double),
                ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double), ("mscale", ctypes.c_double),
                ("mscale_all_dim", ctypes.c_double), ("truncate", ctypes.c_int)]


class DaLayer(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("head_dim", ctypes.c_int), ("num_attention_heads", ctypes.c_int),
                ("num_key_value_heads", ctypes.c_int), ("rotary_dim", ctypes.c_int),
                ("q_norm_w", ctypes.c_void_p), ("k_norm_w", ctypes.c_void_p), ("eps", ctypes.c_double),
                ("window", ctypes.c_int), ("softcap", ctypes.c_float), ("scale", ctypes.c_float),
                ("sinks", ctypes.c_void_p)]


class DaPagedKv(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("n_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("block_table", ctypes.c_void_p), ("num_rows", ctypes.c_int),
                ("max_blocks", ctypes.c_int)]


class DaMlaLayer(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int), ("kv_lora_rank", ctypes.c_int), ("qk_rope_dim", ctypes.c_int),
                ("scale", ctypes.c_float), ("window", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "da_rope_tables_build": (I, [ctypes.POINTER(DaRopeScaling), P, P, I, P, P, P]),
        "da_kv_cache_update": (I, [ctypes.POINTER(DaLayer), P, P, P, I, P, P, P, P, P, P, P, I, I, P]),
        "da_kv_cache_update_rope": (I, [ctypes.POINTER(DaLayer), ctypes.POINTER(DaRopeScaling), P, P, P, I, P, P, P, P,
                                        P, P, I, I, P]),
        "da_kv_cache_update_rope_paged": (I, [ctypes.POINTER(DaLayer), ctypes.POINTER(DaRopeScaling), P, P, P, I, P, P,
                                              P, P, ctypes.c_void_p, P]),
        "da_attn_prefill": (I, [ctypes.POINTER(DaLayer), P, I, P, P, I, I, I, P, P, P, I, P, P, P, Z, P]),
        "da_attn_decode": (I, [ctypes.POINTER(DaLayer), P, P, P, I, I, I, P, P, P, P, P, Z, P]),
        "da_decode_workspace_bytes": (Z, [ctypes.POINTER(DaLayer), I, I]),
        "da_attn_mixed": (I, [ctypes.POINTER(DaLayer), P, P, P, I, I, I, I, P, P, P, I, I, P, P, ctypes.c_double,
                              ctypes.c_double, P, P, Z, P]),
        "da_attn_mixed_prefill_sms": (I, [ctypes.POINTER(DaLayer), I, ctypes.c_double, ctypes.c_double]),
        "da_attn_mixed_paged": (I, [ctypes.POINTER(DaLayer), P, ctypes.POINTER(DaPagedKv), I, I, P, P, P, I, I, P, P,
                                    ctypes.c_double, ctypes.c_double, P, P, Z, P]),
        "da_attn_decode_noalloc": (I, [ctypes.POINTER(DaLayer), P, P, P, I, I, I, P, P, P, P, P]),
        "da_decode_noalloc_max_scratch_bytes": (Z, []),
        "da_kv_cache_update_paged": (I, [ctypes.POINTER(DaLayer), P, P, P, I, P, P, P, P, P,
                                         ctypes.POINTER(DaPagedKv), P]),
        "da_attn_prefill_paged": (I, [ctypes.POINTER(DaLayer), P, I, ctypes.POINTER(DaPagedKv), I, P, P, P, I, P,
                                      P]),
        "da_attn_decode_paged": (I, [ctypes.POINTER(DaLayer), P, ctypes.POINTER(DaPagedKv), I, P, P, P, P, Z, P]),
        "da_decode_workspace_bytes_paged": (Z, [ctypes.POINTER(DaLayer), I, I]),
        "da_mla_cache_update": (I, [ctypes.POINTER(DaMlaLayer), P, P, I, P, P, P, P, P, P, I, I, P]),
        "da_mla_decode": (I, [ctypes.POINTER(DaMlaLayer), P, P, I, I, I, P, P, P, P, Z, P]),
        "da_mla_workspace_bytes": (Z, [ctypes.POINTER(DaMlaLayer), I, I]),
        "da_mla_cache_update_paged": (I, [ctypes.POINTER(DaMlaLayer), P, P, I, P, P, P, P, P,
                                          ctypes.POINTER(DaPagedKv), P]),
        "da_mla_decode_paged": (I, [ctypes.POINTER(DaMlaLayer), P, ctypes.POINTER(DaPagedKv), I, P, P, P, P, Z, P]),
        "da_mla_workspace_bytes_paged": (Z, [ctypes.POINTER(DaMlaLayer), I, I]),
        "da_mla_softmax_scale": (ctypes.c_double, [I, I, ctypes.c_double, ctypes.c_double]),
        "da_qkv_project_update": (I, [ctypes.POINTER(DaLayer), P, P, P, I, I, P, P, P, P, P, P, P, I, I, P]),
        "da_qkv_project_update_paged": (I, [ctypes.POINTER(DaLayer), P, P, P, I, I, P, P, P, P, P,
                                            ctypes.POINTER(DaPagedKv), P]),
        "da_linear": (I, [P, P, P, I, I, I, P, P]),
        "da_block_pool_create": (P, [I, I, I, I, I]),
        "da_block_pool_destroy": (None, [P]),
        "da_block_pool_reserve": (I, [P, I, I, I]),
        "da_block_pool_release": (I, [P, I]),
        "da_block_pool_free_blocks": (I, [P]),
        "da_block_pool_blocks_needed": (I, [P, I, I]),
        "da_block_pool_table": (ctypes.POINTER(ctypes.c_int32), [P]),
        "da_check_device_error": (I, [P]),
        "da_last_error": (ctypes.c_char_p, []),
        "da_version": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def last_error() -> str:
    return LIB.da_last_error().decode()


def version() -> int:
    return int(LIB.da_version())


def _check(rc):
    if rc != DA_OK:
        raise DecAttnError(rc, last_error())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------------------------------ configs

def rope_scaling(theta, rotary_dim, scaling=None, max_position_embeddings=0):
    """DaRopeScaling from config.json's rope_theta and rope_scaling dict (rope_type or type).

    Returns (struct, keepalive) -- keep the second value alive while the struct is in use (it owns the
    LongRoPE factor arrays)."""
    s = dict(scaling or {})
    kind = s.get("rope_type", s.get("type", "default"))
    if kind not in ROPE_KINDS:
        raise DecAttnError(DA_ERR_UNSUPPORTED, f"RoPE type {kind!r} is not implemented")
    rs = DaRopeScaling()
    rs.kind = ROPE_KINDS[kind]
    rs.theta = float(theta)
    rs.rotary_dim = int(rotary_dim)
    rs.factor = float(s.get("factor") or 0.0)
    rs.low_freq_factor = float(s.get("low_freq_factor") or 0.0)
    rs.high_freq_factor = float(s.get("high_freq_factor") or 0.0)
    rs.original_max_position_embeddings = int(s.get("original_max_position_embeddings") or 0)
    rs.max_position_embeddings = int(max_position_embeddings or 0)
    rs.attention_factor = float(s.get("attention_factor") or 0.0)
    rs.beta_fast = float(s.get("beta_fast") or 0.0)
    rs.beta_slow = float(s.get("beta_slow") or 0.0)
    rs.mscale = float(s.get("mscale") or 0.0)
    rs.mscale_all_dim = float(s.get("mscale_all_dim") or 0.0)
    rs.truncate = 1 if s.get("truncate", True) else 0
    keep = []
    if kind == "longrope":
        for name in ("short_factor", "long_factor"):
            vals = [float(x) for x in s[name]]
            if len(vals) != int(rotary_dim) // 2:
                raise DecAttnError(DA_ERR_INVALID_ARG, f"longrope {name} holds {len(vals)} values, rotary_dim/2 = "
                                                       f"{int(rotary_dim) // 2}")
            arr = (ctypes.c_double * len(vals))(*vals)
            keep.append(arr)
            setattr(rs, name, ctypes.cast(arr, ctypes.POINTER(ctypes.c_double)))
    return rs, keep


def layer(dtype, head_dim, num_attention_heads, num_key_value_heads, rotary_dim=None, q_norm_w=None,
          k_norm_w=None, eps=1e-6, window=0, softcap=0.0, scale=0.0, sinks=None):
    """DaLayer for one layer; q_norm_w/k_norm_w are fp32 device tensors [head_dim] or None, sinks an fp32
    device tensor [num_attention_heads] of learned sink logits or None."""
    L = DaLayer()
    L.dtype = DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    L.head_dim = int(head_dim)
    L.num_attention_heads = int(num_attention_heads)
    L.num_key_value_heads = int(num_key_value_heads)
    L.rotary_dim = int(rotary_dim if rotary_dim is not None else head_dim)
    L.q_norm_w = q_norm_w.data_ptr() if q_norm_w is not None else None
    L.k_norm_w = k_norm_w.data_ptr() if k_norm_w is not None else None
    L.eps = float(eps)
    L.window = int(window)
    L.softcap = float(softcap)
    L.scale = float(scale)
    L.sinks = sinks.data_ptr() if sinks is not None else None
    return L


def window_for_layer(config: dict, layer_idx: int) -> int:
    """The layer's sliding window as DecoderConfig.window reads it (page "42. More models", section "What
    differs between model families"): sliding_window if layer_types marks the layer "sliding_attention",
    else 0. Without layer_types, Mistral windows every layer and Qwen2 (use_sliding_window) the layers
    from max_window_layers on."""
    window = config.get("sliding_window") or 0
    types = config.get("layer_types")
    n = config.get("num_hidden_layers", layer_idx + 1)
    if types is None and window:
        kind = config.get("model_type")
        if kind == "mistral":
            types = ["sliding_attention"] * n
        elif kind == "qwen2" and config.get("use_sliding_window"):
            start = config.get("max_window_layers", n)
            types = ["full_attention" if i < start else "sliding_attention" for i in range(n)]
    if not types or "sliding_attention" not in types:
        return 0
    return window if types[layer_idx] == "sliding_attention" else 0


# ------------------------------------------------------------------------------------------ entry points

def rope_tables_build(rs, positions, seq_len, n, cos, sin, stream=None):
    _check(LIB.da_rope_tables_build(ctypes.byref(rs), _ptr(positions), _ptr(seq_len), int(n), _ptr(cos), _ptr(sin),
                                    _stream(stream)))


def kv_cache_update(L, q, k, v, n, rows, positions, cos, sin, q_rot, k_cache, v_cache, num_rows, max_len,
                    stream=None):
    _check(LIB.da_kv_cache_update(ctypes.byref(L), _ptr(q), _ptr(k), _ptr(v), int(n), _ptr(rows), _ptr(positions),
                                  _ptr(cos), _ptr(sin), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), int(num_rows),
                                  int(max_len), _stream(stream)))


def kv_cache_update_rope(L, rs, q, k, v, n, rows, positions, seq_len, q_rot, k_cache, v_cache, num_rows, max_len,
                         stream=None):
    _check(LIB.da_kv_cache_update_rope(ctypes.byref(L), ctypes.byref(rs), _ptr(q), _ptr(k), _ptr(v), int(n), _ptr(rows),
                                       _ptr(positions), _ptr(seq_len), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache),
                                       int(num_rows), int(max_len), _stream(stream)))


def kv_cache_update_rope_paged(L, rs, q, k, v, n, rows, positions, seq_len, q_rot, kv, stream=None):
    _check(LIB.da_kv_cache_update_rope_paged(ctypes.byref(L), ctypes.byref(rs), _ptr(q), _ptr(k), _ptr(v), int(n),
                                             _ptr(rows), _ptr(positions), _ptr(seq_len), _ptr(q_rot),
                                             ctypes.cast(ctypes.pointer(kv), ctypes.c_void_p), _stream(stream)))


def kv_rope_fused_supported(L):
    """Whether da_kv_cache_update_rope takes this layer (bf16, head_dim 128, rotary_dim a multiple of 16)."""
    return L.dtype == DA_BF16 and L.head_dim == 128 and L.rotary_dim % 16 == 0


def attn_prefill(L, q_rot, n_tokens, k_cache, v_cache, num_rows, max_len, n_seqs, q_start, rows, first_pos,
                 max_q_len, key_positions, out, workspace=None, ws_bytes=0, stream=None):
    _check(LIB.da_attn_prefill(ctypes.byref(L), _ptr(q_rot), int(n_tokens), _ptr(k_cache), _ptr(v_cache),
                               int(num_rows), int(max_len), int(n_seqs), _ptr(q_start), _ptr(rows), _ptr(first_pos),
                               int(max_q_len), _ptr(key_positions), _ptr(out), _ptr(workspace), int(ws_bytes),
                               _stream(stream)))


def attn_decode(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, positions, key_positions, out,
                workspace, ws_bytes, stream=None):
    _check(LIB.da_attn_decode(ctypes.byref(L), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), int(num_rows),
                              int(max_len), int(n_seqs), _ptr(rows), _ptr(positions), _ptr(key_positions), _ptr(out),
                              _ptr(workspace), int(ws_bytes), _stream(stream)))


def attn_mixed(L, q_rot, k_cache, v_cache, num_rows, max_len, n_tokens, n_seqs, q_start, chunk_rows, first_pos,
               max_q_len, n_decode, dec_rows, dec_positions, prefill_pairs, decode_keys, out, workspace, ws_bytes,
               stream=None):
    """da_attn_mixed: the chunks' tokens first in q_rot/out, then the decode tokens (see decattn.h)."""
    _check(LIB.da_attn_mixed(ctypes.byref(L), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), int(num_rows), int(max_len),
                             int(n_tokens), int(n_seqs), _ptr(q_start), _ptr(chunk_rows), _ptr(first_pos),
                             int(max_q_len), int(n_decode), _ptr(dec_rows), _ptr(dec_positions), float(prefill_pairs),
                             float(decode_keys), _ptr(out), _ptr(workspace), int(ws_bytes), _stream(stream)))


def attn_mixed_prefill_sms(L, n_sm, prefill_pairs, decode_keys) -> int:
    r = int(LIB.da_attn_mixed_prefill_sms(ctypes.byref(L), int(n_sm), float(prefill_pairs), float(decode_keys)))
    if r < 0:
        raise DecAttnError(r, last_error())
    return r


def attn_mixed_paged(L, q_rot, kv, n_tokens, n_seqs, q_start, chunk_rows, first_pos, max_q_len, n_decode, dec_rows,
                     dec_positions, prefill_pairs, decode_keys, out, workspace, ws_bytes, stream=None):
    _check(LIB.da_attn_mixed_paged(ctypes.byref(L), _ptr(q_rot), ctypes.byref(kv), int(n_tokens), int(n_seqs),
                                   _ptr(q_start), _ptr(chunk_rows), _ptr(first_pos), int(max_q_len), int(n_decode),
                                   _ptr(dec_rows), _ptr(dec_positions), float(prefill_pairs), float(decode_keys),
                                   _ptr(out), _ptr(workspace), int(ws_bytes), _stream(stream)))


def attn_decode_noalloc(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, positions, key_positions, out,
                        stream=None):
    """da_attn_decode without a workspace argument: the library's fixed scratch is used (see decattn.h)."""
    _check(LIB.da_attn_decode_noalloc(ctypes.byref(L), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), int(num_rows),
                                      int(max_len), int(n_seqs), _ptr(rows), _ptr(positions), _ptr(key_positions),
                                      _ptr(out), _stream(stream)))


def decode_noalloc_max_scratch_bytes() -> int:
    return int(LIB.da_decode_noalloc_max_scratch_bytes())


def decode_workspace_bytes(L, n_seqs, max_len) -> int:
    return int(LIB.da_decode_workspace_bytes(ctypes.byref(L), int(n_seqs), int(max_len)))


def paged_kv(k_pool, v_pool, block_table, block_size):
    """DaPagedKv for device pools [n_blocks, Hkv, block_size, d] and an int32 block table [num_rows, max_blocks]
    (keep the tensors alive while the struct is in use)."""
    kv = DaPagedKv()
    kv.k_pool = k_pool.data_ptr()
    kv.v_pool = v_pool.data_ptr()
    kv.n_blocks = int(k_pool.shape[0])
    kv.block_size = int(block_size)
    kv.block_table = block_table.data_ptr()
    kv.num_rows = int(block_table.shape[0])
    kv.max_blocks = int(block_table.shape[1])
    return kv


def kv_cache_update_paged(L, q, k, v, n, rows, positions, cos, sin, q_rot, kv, stream=None):
    _check(LIB.da_kv_cache_update_paged(ctypes.byref(L), _ptr(q), _ptr(k), _ptr(v), int(n), _ptr(rows),
                                        _ptr(positions), _ptr(cos), _ptr(sin), _ptr(q_rot), ctypes.byref(kv),
                                        _stream(stream)))


def attn_prefill_paged(L, q_rot, n_tokens, kv, n_seqs, q_start, rows, first_pos, max_q_len, out, stream=None):
    _check(LIB.da_attn_prefill_paged(ctypes.byref(L), _ptr(q_rot), int(n_tokens), ctypes.byref(kv), int(n_seqs),
                                     _ptr(q_start), _ptr(rows), _ptr(first_pos), int(max_q_len), _ptr(out),
                                     _stream(stream)))


def attn_decode_paged(L, q_rot, kv, n_seqs, rows, positions, out, workspace, ws_bytes, stream=None):
    _check(LIB.da_attn_decode_paged(ctypes.byref(L), _ptr(q_rot), ctypes.byref(kv), int(n_seqs), _ptr(rows),
                                    _ptr(positions), _ptr(out), _ptr(workspace), int(ws_bytes), _stream(stream)))


def decode_workspace_bytes_paged(L, n_seqs, max_positions) -> int:
    return int(LIB.da_decode_workspace_bytes_paged(ctypes.byref(L), int(n_seqs), int(max_positions)))


def mla_softmax_scale(qk_nope_head_dim, qk_rope_head_dim, rope_scaling=None) -> float:
    s = rope_scaling or {}
    return float(LIB.da_mla_softmax_scale(int(qk_nope_head_dim), int(qk_rope_head_dim), float(s.get("factor") or 0.0),
                                          float(s.get("mscale_all_dim") or 0.0)))


def mla_layer(num_heads, scale, kv_lora_rank=512, qk_rope_dim=64, window=0):
    L = DaMlaLayer()
    L.num_heads, L.kv_lora_rank, L.qk_rope_dim = int(num_heads), int(kv_lora_rank), int(qk_rope_dim)
    L.scale, L.window = float(scale), int(window)
    return L


def mla_cache_update(L, latent, k_rope, n, rows, positions, cos, sin, q, cache, num_rows, max_len, stream=None):
    _check(LIB.da_mla_cache_update(ctypes.byref(L), _ptr(latent), _ptr(k_rope), int(n), _ptr(rows), _ptr(positions),
                                   _ptr(cos), _ptr(sin), _ptr(q), _ptr(cache), int(num_rows), int(max_len),
                                   _stream(stream)))


def mla_decode(L, q, cache, num_rows, max_len, n_seqs, rows, positions, out, workspace, ws_bytes, stream=None):
    _check(LIB.da_mla_decode(ctypes.byref(L), _ptr(q), _ptr(cache), int(num_rows), int(max_len), int(n_seqs),
                             _ptr(rows), _ptr(positions), _ptr(out), _ptr(workspace), int(ws_bytes), _stream(stream)))


def mla_workspace_bytes(L, n_seqs, max_len) -> int:
    return int(LIB.da_mla_workspace_bytes(ctypes.byref(L), int(n_seqs), int(max_len)))


def mla_cache_update_paged(L, latent, k_rope, n, rows, positions, cos, sin, q, kv, stream=None):
    _check(LIB.da_mla_cache_update_paged(ctypes.byref(L), _ptr(latent), _ptr(k_rope), int(n), _ptr(rows),
                                         _ptr(positions), _ptr(cos), _ptr(sin), _ptr(q), ctypes.byref(kv),
                                         _stream(stream)))


def mla_decode_paged(L, q, kv, n_seqs, rows, positions, out, workspace, ws_bytes, stream=None):
    _check(LIB.da_mla_decode_paged(ctypes.byref(L), _ptr(q), ctypes.byref(kv), int(n_seqs), _ptr(rows),
                                   _ptr(positions), _ptr(out), _ptr(workspace), int(ws_bytes), _stream(stream)))


def mla_workspace_bytes_paged(L, n_seqs, max_positions) -> int:
    return int(LIB.da_mla_workspace_bytes_paged(ctypes.byref(L), int(n_seqs), int(max_positions)))


def qkv_project_update(L, x, w_qkv, bias, n, hidden, rows, positions, cos, sin, q_rot, k_cache, v_cache, num_rows,
                       max_len, stream=None):
    _check(LIB.da_qkv_project_update(ctypes.byref(L), _ptr(x), _ptr(w_qkv), _ptr(bias), int(n), int(hidden), _ptr(rows),
                                     _ptr(positions), _ptr(cos), _ptr(sin), _ptr(q_rot), _ptr(k_cache), _ptr(v_cache),
                                     int(num_rows), int(max_len), _stream(stream)))


def qkv_project_update_paged(L, x, w_qkv, bias, n, hidden, rows, positions, cos, sin, q_rot, kv, stream=None):
    _check(LIB.da_qkv_project_update_paged(ctypes.byref(L), _ptr(x), _ptr(w_qkv), _ptr(bias), int(n), int(hidden),
                                           _ptr(rows), _ptr(positions), _ptr(cos), _ptr(sin), _ptr(q_rot),
                                           ctypes.byref(kv), _stream(stream)))


def linear(x, w, bias, m, n, k, y, stream=None):
    _check(LIB.da_linear(_ptr(x), _ptr(w), _ptr(bias), int(m), int(n), int(k), _ptr(y), _stream(stream)))


class BlockPool:
    """da_block_pool: host block manager of one layer group's paged pool (see include/decattn.h)."""

    def __init__(self, n_blocks, block_size, num_rows, max_blocks, window=0):
        self._p = LIB.da_block_pool_create(int(n_blocks), int(block_size), int(num_rows), int(max_blocks),
                                           int(window))
        if not self._p:
            raise DecAttnError(DA_ERR_INVALID_ARG, "da_block_pool_create failed")
        self.n_blocks, self.block_size = int(n_blocks), int(block_size)
        self.num_rows, self.max_blocks, self.window = int(num_rows), int(max_blocks), int(window)

    def __del__(self):
        if getattr(self, "_p", None):
            LIB.da_block_pool_destroy(self._p)
            self._p = None

    def reserve(self, row, first_pos, length):
        rc = LIB.da_block_pool_reserve(self._p, int(row), int(first_pos), int(length))
        if rc != DA_OK:
            what = "not enough free blocks" if rc == DA_ERR_OUT_OF_BLOCKS else "invalid row or positions"
            raise DecAttnError(rc, f"reserve(row={row}, first_pos={first_pos}, length={length}): {what}")

    def release(self, row):
        if LIB.da_block_pool_release(self._p, int(row)) != DA_OK:
            raise DecAttnError(DA_ERR_INVALID_ARG, f"release(row={row}): invalid row")

    @property
    def free_blocks(self):
        return int(LIB.da_block_pool_free_blocks(self._p))

    def blocks_needed(self, first_pos, length):
        return int(LIB.da_block_pool_blocks_needed(self._p, int(first_pos), int(length)))

    def table(self):
        """A copy of the host block table, int32 [num_rows, max_blocks]."""
        import numpy as np
        ptr = LIB.da_block_pool_table(self._p)
        arr = np.ctypeslib.as_array(ptr, shape=(self.num_rows * self.max_blocks,)).copy()
        return torch.from_numpy(arr).reshape(self.num_rows, self.max_blocks)


def check_device_error(stream=None):
    _check(LIB.da_check_device_error(_stream(stream)))
