"""One layer's attention step through the C ABI: norm/rope/cache write -> attention.

``AttentionStep`` owns the per-call buffers (cos/sin tables, q_rot, out, decode workspace) that the caller
must provide to the library, allocated once with torch; ``run()`` only enqueues the library's kernels.
Prefill chunks and decode tokens of one batch go to da_attn_prefill and da_attn_decode respectively, or
together to da_attn_mixed when the batch holds both (the library may then run the two side by side),
after one cache update for all tokens: da_kv_cache_update_rope (cos/sin formed in the kernel) where the layer
allows it (bf16, head_dim 128, rotary_dim a multiple of 16), else da_rope_tables_build + da_kv_cache_update.
"""
from __future__ import annotations

import math

import torch

from . import _abi, work


def rotary_dim_of(head_dim, partial_rotary_factor):
    r = int(round(head_dim * partial_rotary_factor))
    if r <= 0 or r % 2 or r > head_dim:
        raise ValueError(f"rotary dim {r} must be even and in (0, {head_dim}]")
    return r


class AttentionStep:
    """Buffers and C structs for one LayerCall (see decoder_attention_gb300.inputs)."""

    def __init__(self, call, device=None, fused_rope=None):
        dev = torch.device(device) if device is not None else call.q.device
        self.call = c = call
        self.device = dev
        self.rot = rotary_dim_of(c.head_dim, c.partial_rotary_factor)
        self.rs, self._keep = _abi.rope_scaling(c.rope_theta, self.rot, c.rope_scaling, c.max_position_embeddings)
        self.q_norm_w = c.q_norm_w.to(dev, torch.float32).contiguous() if c.q_norm_w is not None else None
        self.k_norm_w = c.k_norm_w.to(dev, torch.float32).contiguous() if c.k_norm_w is not None else None
        self.sinks = c.sinks.to(dev, torch.float32).contiguous() if c.sinks is not None else None
        self.L = _abi.layer(c.dtype, c.head_dim, c.num_attention_heads, c.num_key_value_heads, self.rot,
                            self.q_norm_w, self.k_norm_w, c.eps, c.window, c.softcap, 0.0, self.sinks)
        # fused_rope: None = whenever the layer allows it; False = the tables and the update as two calls
        self.fused_rope = _abi.kv_rope_fused_supported(self.L) if fused_rope is None else bool(fused_rope)
        n = c.n_tokens
        self.cos = torch.empty((max(n, 1), self.rot // 2), dtype=torch.float32, device=dev)
        self.sin = torch.empty_like(self.cos)
        self.q_rot = torch.empty_like(c.q)
        self.out = torch.empty_like(c.q)
        self.ws_bytes = 0
        self.workspace = None
        if c.n_decode:
            self.ws_bytes = _abi.decode_workspace_bytes(self.L, c.n_decode, c.max_len)
            if self.ws_bytes:
                self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        # host hints of a mixed batch's two parts for da_attn_mixed: visible (query, key) pairs of one query head
        # over the chunks, visible keys over the decode tokens (read once here from the call's metadata)
        self.hint_pairs = self.hint_keys = 0.0
        if c.n_prefill and c.n_decode:
            w = work.layer_call_work(c)
            self.hint_pairs = w["prefill_pairs"] / c.num_attention_heads
            self.hint_keys = float(w["decode_keys"])

    # -- the three stages, separately callable for timing ------------------------------------------
    def rope(self, stream=None):
        """cos/sin tables (the two-call form needs them; the fused update forms them itself)."""
        c = self.call
        _abi.rope_tables_build(self.rs, c.tok_pos, c.tok_seq_len, c.n_tokens, self.cos, self.sin, stream)

    def update(self, stream=None):
        """Norm, RoPE and the cache write for every token: one fused call, or the tables and the update."""
        if not self.fused_rope:
            self.rope(stream)
        self.cache_update(stream)

    def cache_update(self, stream=None):
        c = self.call
        if self.fused_rope:
            _abi.kv_cache_update_rope(self.L, self.rs, c.q, c.k, c.v, c.n_tokens, c.tok_rows, c.tok_pos, c.tok_seq_len,
                                      self.q_rot, c.k_cache, c.v_cache, c.num_rows, c.max_len, stream)
        else:
            _abi.kv_cache_update(self.L, c.q, c.k, c.v, c.n_tokens, c.tok_rows, c.tok_pos, self.cos, self.sin,
                                 self.q_rot, c.k_cache, c.v_cache, c.num_rows, c.max_len, stream)

    def prefill(self, stream=None):
        c = self.call
        if c.n_prefill:
            _abi.attn_prefill(self.L, self.q_rot, c.n_prefill, c.k_cache, c.v_cache, c.num_rows, c.max_len,
                              len(c.pf_rows), c.q_start, c.pf_rows, c.pf_first_pos, c.max_q_len, None, self.out,
                              None, 0, stream)

    def decode(self, stream=None):
        c = self.call
        if c.n_decode:
            _abi.attn_decode(self.L, self.q_rot[c.n_prefill:], c.k_cache, c.v_cache, c.num_rows, c.max_len,
                             c.n_decode, c.dec_rows, c.dec_pos, None, self.out[c.n_prefill:], self.workspace,
                             self.ws_bytes, stream)

    def attend(self, stream=None):
        """Attention of every token: one da_attn_mixed call when the batch has chunks and decode tokens."""
        c = self.call
        if c.n_prefill and c.n_decode:
            self.mixed(stream)
        else:
            self.prefill(stream)
            self.decode(stream)

    def mixed(self, stream=None):
        c = self.call
        _abi.attn_mixed(self.L, self.q_rot, c.k_cache, c.v_cache, c.num_rows, c.max_len, c.n_prefill, len(c.pf_rows),
                        c.q_start, c.pf_rows, c.pf_first_pos, c.max_q_len, c.n_decode, c.dec_rows, c.dec_pos,
                        self.hint_pairs, self.hint_keys, self.out, self.workspace, self.ws_bytes, stream)

    def run(self, stream=None):
        self.update(stream)
        self.attend(stream)
        return self.out

    def kernel_launches(self):
        """Kernels one run() enqueues (rope tables unless fused, cache update, prefill, decode + merge)."""
        c = self.call
        n = (1 if c.n_tokens else 0) * (1 if self.fused_rope else 2)
        if c.n_prefill:
            n += 1
        if c.n_decode:
            n += 2 if self.workspace is not None else 1
        return n


class PagedAttentionStep(AttentionStep):
    """AttentionStep over a paged KV pool: k_pool/v_pool [n_blocks, Hkv, block_size, d] and an int32 block
    table [num_rows, max_blocks] on the device stand in for the call's contiguous caches."""

    def __init__(self, call, k_pool, v_pool, block_table, block_size, device=None, fused_rope=None):
        super().__init__(call, device, fused_rope)
        self.k_pool, self.v_pool, self.block_table = k_pool, v_pool, block_table
        self.block_size = int(block_size)
        self.kv = _abi.paged_kv(k_pool, v_pool, block_table, block_size)
        self.max_positions = int(block_table.shape[1]) * self.block_size
        self.ws_bytes = 0
        self.workspace = None
        c = call
        if c.n_decode:
            self.ws_bytes = _abi.decode_workspace_bytes_paged(self.L, c.n_decode, self.max_positions)
            if self.ws_bytes:
                self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)

    def cache_update(self, stream=None):
        c = self.call
        if self.fused_rope:
            _abi.kv_cache_update_rope_paged(self.L, self.rs, c.q, c.k, c.v, c.n_tokens, c.tok_rows, c.tok_pos,
                                            c.tok_seq_len, self.q_rot, self.kv, stream)
        else:
            _abi.kv_cache_update_paged(self.L, c.q, c.k, c.v, c.n_tokens, c.tok_rows, c.tok_pos, self.cos, self.sin,
                                       self.q_rot, self.kv, stream)

    def prefill(self, stream=None):
        c = self.call
        if c.n_prefill:
            _abi.attn_prefill_paged(self.L, self.q_rot, c.n_prefill, self.kv, len(c.pf_rows), c.q_start, c.pf_rows,
                                    c.pf_first_pos, c.max_q_len, self.out, stream)

    def decode(self, stream=None):
        c = self.call
        if c.n_decode:
            _abi.attn_decode_paged(self.L, self.q_rot[c.n_prefill:], self.kv, c.n_decode, c.dec_rows, c.dec_pos,
                                   self.out[c.n_prefill:], self.workspace, self.ws_bytes, stream)

    def mixed(self, stream=None):
        c = self.call
        _abi.attn_mixed_paged(self.L, self.q_rot, self.kv, c.n_prefill, len(c.pf_rows), c.q_start, c.pf_rows,
                              c.pf_first_pos, c.max_q_len, c.n_decode, c.dec_rows, c.dec_pos, self.hint_pairs,
                              self.hint_keys, self.out, self.workspace, self.ws_bytes, stream)



class MlaDecodeStep:
    """Buffers and C structs for one MLA decode step (see decoder_attention_gb300.inputs.MlaCall): rope tables
    for the 64 rotary features, the cache update (rows written, queries' rotary part rotated in place) and the
    absorbed decode. Over a paged pool when k_pool and block_table are given."""

    def __init__(self, call, k_pool=None, block_table=None, block_size=0):
        c = self.call = call
        dev = c.q.device
        self.rs, self._keep = _abi.rope_scaling(c.rope_theta, c.qk_rope_head_dim, c.rope_scaling,
                                                c.max_position_embeddings)
        self.scale = _abi.mla_softmax_scale(c.qk_nope_head_dim, c.qk_rope_head_dim, c.rope_scaling)
        self.L = _abi.mla_layer(c.num_heads, self.scale, window=c.window)
        S = c.n_seqs
        self.cos = torch.empty((max(S, 1), c.qk_rope_head_dim // 2), dtype=torch.float32, device=dev)
        self.sin = torch.empty_like(self.cos)
        self.q_rot = c.q.clone()
        self.out = torch.empty((S, c.num_heads, 512), dtype=c.q.dtype, device=dev)
        self.kv = None
        if k_pool is not None:
            self.k_pool, self.block_table = k_pool, block_table
            self.kv = _abi.paged_kv(k_pool, k_pool, block_table, block_size)
            self.ws_bytes = _abi.mla_workspace_bytes_paged(self.L, S, int(block_table.shape[1]) * int(block_size))
        else:
            self.ws_bytes = _abi.mla_workspace_bytes(self.L, S, c.max_len)
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)

    def rope(self, stream=None):
        c = self.call
        _abi.rope_tables_build(self.rs, c.positions, c.seq_len, c.n_seqs, self.cos, self.sin, stream)

    def cache_update(self, stream=None):
        c = self.call
        self.q_rot.copy_(c.q)
        if self.kv is not None:
            _abi.mla_cache_update_paged(self.L, c.latent, c.k_rope, c.n_seqs, c.rows, c.positions, self.cos, self.sin,
                                        self.q_rot, self.kv, stream)
        else:
            _abi.mla_cache_update(self.L, c.latent, c.k_rope, c.n_seqs, c.rows, c.positions, self.cos, self.sin,
                                  self.q_rot, c.cache, c.num_rows, c.max_len, stream)


    def update(self, stream=None):
        """The rotary tables, then the cache rows and the queries' rotated part."""
        self.rope(stream)
        self.cache_update(stream)
    def decode(self, stream=None):
        c = self.call
        if self.kv is not None:
            _abi.mla_decode_paged(self.L, self.q_rot, self.kv, c.n_seqs, c.rows, c.positions, self.out,
                                  self.workspace, self.ws_bytes, stream)
        else:
            _abi.mla_decode(self.L, self.q_rot, c.cache, c.num_rows, c.max_len, c.n_seqs, c.rows, c.positions,
                            self.out, self.workspace, self.ws_bytes, stream)

    def run(self, stream=None):
        self.rope(stream)
        self.cache_update(stream)
        self.decode(stream)
        return self.out

    def kernel_launches(self):
        return 4 if self.call.n_seqs else 0     # rope tables, cache update, decode, merge
