"""Plain fp64 CPU oracle for the attention step of a rotary grouped-query decoder layer.

THIS MODULE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py`` may import it. The CUDA library never calls it and shares no code with it.

It restates, in float64 numpy and in the order the pages give them, the steps that the
``DecoderAttention.forward`` method of the page "42. More models: a registry, scaled RoPE, sliding
windows and latent attention" (inference.shantanugoel.com, section "What differs between model
families") performs between the q/k/v projections and o_proj:

    optional per-head q/k RMSNorm -> RoPE on q and k -> cache.update at (rows, positions)
    -> optional window mask -> causal GQA softmax attention (optional logit soft-cap)

Where the pages leave a step open the oracle takes one reading; each is named where it is used:

  R1  partial rotation: r = round(d * partial_rotary_factor) rotated dims, frequency exponent 2i/r,
      split-half pairs (i, i + r/2) inside the first r dims.
  R2  LongRoPE: per-pair divisors of the base frequencies; the long table is used for every token of a
      sequence whose total length in the step exceeds original_max_position_embeddings.
  R3  the attention factor multiplies cos and sin only; dims past r pass through unscaled.
  R4  query head h reads KV head floor(h / G), G = Hq / Hkv (contiguous groups).
  R5  soft-cap = cap * tanh(z / cap) on the scaled logit, before masking; cap = 0 means off.
  R7  a query with no allowed key gets output 0.
  R8  a window of w admits w keys including the query's own: key position j is allowed for a query at
      position p iff j <= p and p - j <= w - 1 (w = 0: no window).
  R17 paged cache: position p of cache row `row` lives in pool block block_table[row, p // block_size] at
      offset p % block_size (page 1 "Sliding windows" names the engine's blocks and block tables but not
      their layout); a block that lies wholly before the first position a call's oldest query can see is
      never read, so it may be recycled (its table slot -1).
  R16 a learned sink (page "Model resolution", gpt_oss entry: one extra logit per head in every query's
      softmax whose share is dropped) is a logit in the units of the scaled scores, after any soft-cap and
      not capped itself, seen by every query whatever its window; its probability multiplies no value.

Parity pins for every function live in ``tests/test_oracle_*.py``; none is left unpinned.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------------------------------
# Frequencies  (page 1, section "Scaled RoPE", function rope_inv_freq)
# --------------------------------------------------------------------------------------------------

def rotary_dim(head_dim: int, partial_rotary_factor: float = 1.0) -> int:
    """Number of rotated dims of a head (reading R1).

    "Model resolution" (Overview) says that under partial_rotary_factor only that share of each
    head rotates. We round d * factor to the nearest integer; it must be even.
    """
    r = int(round(head_dim * partial_rotary_factor))
    if r <= 0 or r % 2 or r > head_dim:
        raise ValueError(f"rotary dim {r} (head_dim {head_dim}, factor {partial_rotary_factor}) must be even and in (0, d]")
    return r


def rope_inv_freq(rot_dim: int, theta: float, scaling: dict | None = None,
                  max_position_embeddings: int | None = None, seq_len: int | None = None):
    """Rotation frequency of each of the rot_dim/2 feature pairs and the attention factor.

    Page 1, "Scaled RoPE": base_i = theta^(-2i/dim) for the pairs i < dim/2 (dim = the rotated width,
    reading R1), then by rope_type (or type):
      default  base, factor 1
      linear   every frequency divided by `factor`
      llama3   pairs whose wavelength 2*pi/base_i exceeds old/low_freq_factor are divided by `factor`,
               the ones below old/high_freq_factor are kept, and in between the frequency is the blend
               (1 - smooth) * base/factor + smooth * base with smooth = (old/wavelength - low)/(high - low)
      longrope (reading R2) divisors: base / short_factor while seq_len <= original_max_position_embeddings,
               base / long_factor past it; the attention factor is `attention_factor` when given, else
               sqrt(1 + ln s / ln original) with s = max_position_embeddings / original (1 when s <= 1)
      yarn     ramp over pair index between the pairs that turn beta_fast and beta_slow times over the
               original context; attention factor 0.1 ln s + 1 (or the mscale ratio, or as given)
    Returns (inv_freq float64 [rot_dim/2], attention_factor float).
    """
    if rot_dim <= 0 or rot_dim % 2:
        raise ValueError(f"rotary dim must be positive and even, got {rot_dim}")
    i = np.arange(rot_dim // 2, dtype=F64)
    base = 1.0 / np.power(F64(theta), 2.0 * i / rot_dim)
    s = scaling or {}
    kind = s.get("rope_type", s.get("type", "default"))
    if kind == "default":
        return base, 1.0
    factor = s.get("factor")
    if kind == "linear":
        return base / factor, 1.0
    if kind == "llama3":
        old = float(s["original_max_position_embeddings"])
        low, high = float(s["low_freq_factor"]), float(s["high_freq_factor"])
        wavelen = 2.0 * math.pi / base
        scaled = np.where(wavelen > old / low, base / factor, base)
        smooth = (old / wavelen - low) / (high - low)
        medium = (wavelen <= old / low) & (wavelen >= old / high)
        return np.where(medium, (1.0 - smooth) * base / factor + smooth * base, scaled), 1.0
    if kind == "longrope":
        old = int(s["original_max_position_embeddings"])
        short = np.asarray(s["short_factor"], dtype=F64)
        long_ = np.asarray(s["long_factor"], dtype=F64)
        if short.shape != (rot_dim // 2,) or long_.shape != (rot_dim // 2,):
            raise ValueError("longrope factor lists must hold rot_dim/2 values each")
        if seq_len is None:
            raise ValueError("longrope needs the sequence length to choose its table")
        ext = long_ if seq_len > old else short
        af = s.get("attention_factor")
        if af is None:
            mpe = max_position_embeddings if max_position_embeddings else old
            ratio = mpe / old
            af = 1.0 if ratio <= 1.0 else math.sqrt(1.0 + math.log(ratio) / math.log(old))
        return base / ext, float(af)
    if kind == "yarn":
        old = float(s["original_max_position_embeddings"])
        factor = factor or (max_position_embeddings / old)

        def mscale(scale, m=1.0):
            return 1.0 if scale <= 1 else 0.1 * m * math.log(scale) + 1.0

        af = s.get("attention_factor")
        if af is None:
            if s.get("mscale") and s.get("mscale_all_dim"):
                af = mscale(factor, s["mscale"]) / mscale(factor, s["mscale_all_dim"])
            else:
                af = mscale(factor)

        def pair_turning(rotations):
            # the (fractional) pair index whose wavelength fits `rotations` times into `old`
            return rot_dim * math.log(old / (rotations * 2.0 * math.pi)) / (2.0 * math.log(theta))

        lo = pair_turning(s.get("beta_fast") or 32)
        hi = pair_turning(s.get("beta_slow") or 1)
        if s.get("truncate", True):
            lo, hi = math.floor(lo), math.ceil(hi)
        lo, hi = max(lo, 0), min(hi, rot_dim - 1)
        span = (hi - lo) if hi != lo else 0.001
        ramp = np.clip((i - lo) / span, 0.0, 1.0)
        keep = 1.0 - ramp
        return base / factor * (1.0 - keep) + base * keep, float(af)
    raise ValueError(f"RoPE type {kind!r} is not implemented")


# --------------------------------------------------------------------------------------------------
# Tables, norm, rotation  (page 1 "Scaled RoPE" rope_tables; page 3 §3.2 RMSNorm and §4 Rotary)
# --------------------------------------------------------------------------------------------------

def rope_tables(positions, inv_freq, attention_factor):
    """cos and sin [N, r/2] of angle p * inv_freq_i, each times the attention factor.

    Page 1, rope_tables: angles = positions * inv_freq, cos and sin times the factor. The page then
    concatenates the angles with themselves to width r; we keep the r/2 distinct columns, which is the
    same table (page 3 §4 keeps the half tables too). The page's cast to the activation dtype is not
    reproduced: the oracle stays in float64.
    """
    p = np.asarray(positions, dtype=F64)[:, None]
    ang = p * np.asarray(inv_freq, dtype=F64)[None, :]
    return np.cos(ang) * attention_factor, np.sin(ang) * attention_factor


def rms_norm(x, weight, eps):
    """x / sqrt(mean over the last axis of x^2 + eps) * weight (page 3 §3.2 RMSNorm; page 1 q_norm/k_norm
    act per head over head_dim). The page's intermediate cast back to the input dtype is not reproduced."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(weight, dtype=F64)


def apply_rope(x, cos, sin):
    """Rotate split-half pairs (i, i + r/2), i < r/2, of the first r dims; the rest pass through.

    Page 3 §4 (Rotary.forward): x1, x2 halves -> [x1 cos - x2 sin, x1 sin + x2 cos]; page 1 says the
    engine's apply_rope uses the same split-half pairing. x [..., T, d] with cos/sin broadcastable to
    [..., T, r/2]; r = 2 * cos.shape[-1] (reading R1, R3).
    """
    x = np.asarray(x, dtype=F64)
    half = cos.shape[-1]
    r = 2 * half
    x1, x2, rest = x[..., :half], x[..., half:r], x[..., r:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin, rest], axis=-1)


# --------------------------------------------------------------------------------------------------
# Mask and attention  (page 1 "Sliding windows" and DecoderAttention.forward; page 3 §2.3, §3.4)
# --------------------------------------------------------------------------------------------------

def window_allowed(q_pos, k_pos, window):
    """Boolean [T, S]: key at position k_pos[j] is visible to the query at q_pos[t].

    Causal over positions (the key is not after the query), and with a window w > 0 the key may be at
    most w - 1 positions back (page 1, "Sliding windows"; reading R8). Negative key positions mark empty
    slots and are never visible.
    """
    qp = np.asarray(q_pos, dtype=np.int64)[:, None]
    kp = np.asarray(k_pos, dtype=np.int64)[None, :]
    ok = (kp >= 0) & (kp <= qp)
    if window:
        ok &= (qp - kp) <= (window - 1)
    return ok


def causal_attention(q, k, v, q_pos, k_pos, window=0, softcap=0.0, scale=None, sinks=None):
    """GQA softmax attention for one cache row.

    q [T, Hq, d] (already rotated), k/v [Hkv, S, d], q_pos [T], k_pos [S] (negative = empty slot).
    For query head h the KV head is floor(h / G) (reading R4). Logits z = scale * q.k with scale
    1/sqrt(d) by default (page 3 §3.4); soft-capped by cap * tanh(z / cap) when softcap > 0 (R5);
    softmax over the allowed keys only (page 3 §2.3: a masked logit is -inf, probability 0); output
    0 for a query that sees no key (R7). With sinks [Hq], head h's softmax also takes the logit sinks[h],
    whose probability is dropped (R16). Returns float64 [T, Hq, d].
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    T, hq, d = q.shape
    hkv = k.shape[0]
    if hq % hkv:
        raise ValueError("num_attention_heads must be a multiple of num_key_value_heads")
    group = hq // hkv
    if scale is None or scale == 0:
        scale = 1.0 / math.sqrt(d)
    allowed = window_allowed(q_pos, k_pos, window)                       # [T, S]
    out = np.zeros((T, hq, d), dtype=F64)
    for h in range(hq):
        g = h // group
        z = scale * (q[:, h, :] @ k[g].T)                                # [T, S]
        if softcap and softcap > 0:
            z = softcap * np.tanh(z / softcap)
        z = np.where(allowed, z, -np.inf)
        zmax = np.max(z, axis=1, keepdims=True)
        has_key = np.isfinite(zmax[:, 0])
        sink = None if sinks is None else float(sinks[h])
        if sink is not None:
            zmax = np.maximum(zmax, sink)
        zmax = np.where(np.isfinite(zmax), zmax, 0.0)
        e = np.where(allowed, np.exp(z - zmax), 0.0)
        den = e.sum(axis=1, keepdims=True)
        if sink is not None:
            den = den + np.exp(sink - zmax)
        w = np.divide(e, den, out=np.zeros_like(e), where=den > 0)
        o = w @ v[g]
        o[~has_key] = 0.0
        out[:, h, :] = o
    return out


# --------------------------------------------------------------------------------------------------
# The step as the library's entry points present it
# --------------------------------------------------------------------------------------------------

@dataclass
class Layer:
    """The per-layer switches the step reads (page 1, DecoderConfig and DecoderAttention.__init__)."""
    head_dim: int
    num_attention_heads: int
    num_key_value_heads: int
    rotary_dim: int
    q_norm_w: np.ndarray | None = None      # None: no q/k norm ("absent, not identity")
    k_norm_w: np.ndarray | None = None
    eps: float = 1e-6
    window: int = 0                         # 0: full attention
    softcap: float = 0.0                    # 0: off
    scale: float = 0.0                      # 0: 1/sqrt(head_dim)
    sinks: np.ndarray | None = None         # [Hq] learned sink logits (R16), or None


@dataclass
class RopeSpec:
    theta: float
    scaling: dict | None = None
    max_position_embeddings: int | None = None
    extra: dict = field(default_factory=dict)


def rope_tables_for_tokens(spec: RopeSpec, rot_dim: int, positions, seq_len=None):
    """cos/sin [N, r/2] for each token; LongRoPE picks its table per token's sequence length (R2)."""
    positions = np.asarray(positions, dtype=np.int64)
    n = positions.shape[0]
    cos = np.zeros((n, rot_dim // 2), dtype=F64)
    sin = np.zeros((n, rot_dim // 2), dtype=F64)
    lens = np.asarray(seq_len, dtype=np.int64) if seq_len is not None else np.full(n, -1)
    # tokens that share a sequence length share a table
    for L in np.unique(lens):
        sel = lens == L
        inv, af = rope_inv_freq(rot_dim, spec.theta, spec.scaling, spec.max_position_embeddings,
                                int(L) if L >= 0 else None)
        c, s = rope_tables(positions[sel], inv, af)
        cos[sel], sin[sel] = c, s
    return cos, sin


def kv_cache_update(layer: Layer, q, k, v, rows, positions, cos, sin, k_cache, v_cache):
    """Norm (optional), rotate q and k, and write k_rot and v at (rows[t], :, positions[t]).

    Page 1, DecoderAttention.forward: q_norm/k_norm before apply_rope, then cache.update(layer, k, v,
    positions, rows); page 3 §3.3 KVCache.update writes the new keys at their positions. q [N, Hq, d],
    k/v [N, Hkv, d], cos/sin [N, r/2]; k_cache/v_cache [R, Hkv, M, d] float64, updated in place.
    Returns q_rot [N, Hq, d] float64.
    """
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    if layer.q_norm_w is not None:
        q = rms_norm(q, layer.q_norm_w, layer.eps)
        k = rms_norm(k, layer.k_norm_w, layer.eps)
    c = np.asarray(cos, dtype=F64)[:, None, :]
    s = np.asarray(sin, dtype=F64)[:, None, :]
    q_rot = apply_rope(q, c, s)
    k_rot = apply_rope(k, c, s)
    for t in range(q.shape[0]):
        k_cache[rows[t], :, positions[t], :] = k_rot[t]
        v_cache[rows[t], :, positions[t], :] = np.asarray(v[t], dtype=F64)
    return q_rot


def attn_prefill(layer: Layer, q_rot, k_cache, v_cache, q_start, rows, first_pos, key_positions=None):
    """Prefill chunks: sequence b owns tokens q_start[b]..q_start[b+1]-1 at positions first_pos[b] + i.

    Each chunk sees the keys of its cache row: slots 0 .. first_pos[b] + n_b - 1 with slot index =
    position, or, with key_positions [R, M], every slot whose position is not negative (page 1,
    DecoderAttention.forward: kp = key_positions or arange, qp = positions).
    """
    q_rot = np.asarray(q_rot, dtype=F64)
    out = np.zeros_like(q_rot)
    for b in range(len(rows)):
        t0, t1 = int(q_start[b]), int(q_start[b + 1])
        if t1 <= t0:
            continue
        qp = int(first_pos[b]) + np.arange(t1 - t0)
        kv_len = int(first_pos[b]) + (t1 - t0)
        row = int(rows[b])
        if key_positions is None:
            kp = np.arange(kv_len)
            kk, vv = k_cache[row, :, :kv_len], v_cache[row, :, :kv_len]
        else:
            kp = np.asarray(key_positions[row], dtype=np.int64)
            kk, vv = k_cache[row], v_cache[row]
        out[t0:t1] = causal_attention(q_rot[t0:t1], kk, vv, qp, kp, layer.window, layer.softcap, layer.scale,
                                      layer.sinks)
    return out


def attn_decode(layer: Layer, q_rot, k_cache, v_cache, rows, positions, key_positions=None):
    """One new token per sequence s at position positions[s] of cache row rows[s]: it sees slots
    0..positions[s] (its own key was just written), or the key_positions form as in attn_prefill."""
    q_rot = np.asarray(q_rot, dtype=F64)
    out = np.zeros_like(q_rot)
    for s in range(len(rows)):
        p, row = int(positions[s]), int(rows[s])
        if key_positions is None:
            lo = 0
            if layer.window:
                lo = max(0, p - layer.window + 1)   # keys before lo are masked anyway; skip reading them
            kp = np.arange(lo, p + 1)
            kk, vv = k_cache[row, :, lo:p + 1], v_cache[row, :, lo:p + 1]
        else:
            kp = np.asarray(key_positions[row], dtype=np.int64)
            kk, vv = k_cache[row], v_cache[row]
        out[s:s + 1] = causal_attention(q_rot[s:s + 1], kk, vv, [p], kp, layer.window, layer.softcap, layer.scale,
                                        layer.sinks)
    return out


def attn_decode_one(layer: Layer, q_vec, k_row, v_row, p):
    """Output of one query vector set q_vec [Hq, d] at position p against k_row/v_row [Hkv, >=p+1, d]
    (slot = position). Used to check sampled outputs of full-size workloads one by one."""
    lo = max(0, p - layer.window + 1) if layer.window else 0
    kp = np.arange(lo, p + 1)
    return causal_attention(np.asarray(q_vec, dtype=F64)[None], k_row[:, lo:p + 1], v_row[:, lo:p + 1],
                            [p], kp, layer.window, layer.softcap, layer.scale, layer.sinks)[0]


# --------------------------------------------------------------------------------------------------
# Paged KV cache  (page 1 "Sliding windows": the engine's cache is a pool of fixed-size blocks that each
# request maps through its own block table, and blocks that every query has moved past can be recycled)
# --------------------------------------------------------------------------------------------------

def paged_view(pool, block_table, block_size, row, lo, hi):
    """Keys (or values) of positions lo .. hi-1 of cache row `row`, [Hkv, hi - lo, d] float64.

    pool [n_blocks, Hkv, block_size, d]; block_table [R, max_blocks] int (-1 = no block). Position p of the
    row lives at pool[block_table[row, p // block_size], :, p % block_size]. A position whose block is not
    mapped raises: nothing the step reads may be unmapped."""
    pool = np.asarray(pool)
    hkv, d = pool.shape[1], pool.shape[3]
    out = np.empty((hkv, max(hi - lo, 0), d), dtype=F64)
    for p in range(lo, hi):
        b = int(block_table[row][p // block_size])
        if b < 0:
            raise ValueError(f"position {p} of row {row} has no block")
        out[:, p - lo] = pool[b, :, p % block_size]
    return out


def kv_cache_update_paged(layer: Layer, q, k, v, rows, positions, cos, sin, k_pool, v_pool, block_table,
                          block_size):
    """kv_cache_update with the cache slot of (row, position) found through the row's block table."""
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    if layer.q_norm_w is not None:
        q = rms_norm(q, layer.q_norm_w, layer.eps)
        k = rms_norm(k, layer.k_norm_w, layer.eps)
    c = np.asarray(cos, dtype=F64)[:, None, :]
    s = np.asarray(sin, dtype=F64)[:, None, :]
    q_rot = apply_rope(q, c, s)
    k_rot = apply_rope(k, c, s)
    for t in range(q.shape[0]):
        p = int(positions[t])
        b = int(block_table[rows[t]][p // block_size])
        if b < 0:
            raise ValueError(f"position {p} of row {rows[t]} has no block")
        k_pool[b, :, p % block_size, :] = k_rot[t]
        v_pool[b, :, p % block_size, :] = np.asarray(v[t], dtype=F64)
    return q_rot


def _first_visible(first_pos, window):
    """Oldest position any query from first_pos on can see: keys before it are masked for all of them."""
    return max(0, first_pos - window + 1) if window else 0


def attn_prefill_paged(layer: Layer, q_rot, k_pool, v_pool, block_table, block_size, q_start, rows, first_pos):
    """attn_prefill over a paged cache: chunk b sees positions lo .. first_pos[b] + n_b - 1 of its row, lo
    the first position its oldest query can see (blocks wholly before lo may be unmapped)."""
    q_rot = np.asarray(q_rot, dtype=F64)
    out = np.zeros_like(q_rot)
    for b in range(len(rows)):
        t0, t1 = int(q_start[b]), int(q_start[b + 1])
        if t1 <= t0:
            continue
        fp = int(first_pos[b])
        qp = fp + np.arange(t1 - t0)
        kv_len = fp + (t1 - t0)
        lo = _first_visible(fp, layer.window)
        row = int(rows[b])
        kk = paged_view(k_pool, block_table, block_size, row, lo, kv_len)
        vv = paged_view(v_pool, block_table, block_size, row, lo, kv_len)
        out[t0:t1] = causal_attention(q_rot[t0:t1], kk, vv, qp, np.arange(lo, kv_len), layer.window, layer.softcap,
                                      layer.scale, layer.sinks)
    return out


def attn_decode_paged(layer: Layer, q_rot, k_pool, v_pool, block_table, block_size, rows, positions):
    """attn_decode over a paged cache: the token at position p of row rows[s] sees positions lo .. p."""
    q_rot = np.asarray(q_rot, dtype=F64)
    out = np.zeros_like(q_rot)
    for s in range(len(rows)):
        p, row = int(positions[s]), int(rows[s])
        lo = _first_visible(p, layer.window)
        kk = paged_view(k_pool, block_table, block_size, row, lo, p + 1)
        vv = paged_view(v_pool, block_table, block_size, row, lo, p + 1)
        out[s:s + 1] = causal_attention(q_rot[s:s + 1], kk, vv, [p], np.arange(lo, p + 1), layer.window,
                                        layer.softcap, layer.scale, layer.sinks)
    return out

