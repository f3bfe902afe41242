"""Seeded synthetic workloads for the attention step.

This module draws random numbers and lays out bookkeeping (rows, positions, chunk offsets); it holds
none of the step's arithmetic, so both the CUDA path and the CPU oracle can take their inputs from it.

Five workloads, shaped like the model families the pages discuss (page 1, "What differs between model
families" and "Sliding windows"; "Model resolution", Overview, for Phi/longrope/partial rotation and Gemma 2
soft-capping):

  1 tiny_prefill_fp32        B=1 x 128 tokens, Hq=4, Hkv=2, d=64, fp32, theta 1e4, full causal
  2 qwen3_8b_prefill         B=4 x 2048 tokens, Hq=32, Hkv=8, d=128, bf16, q/k RMSNorm, theta 1e6
  3 mistral_swa_decode       64 sequences, contexts U[1024, 32768], window 4096, theta 1e6
  4 llama31_8b_long_decode   16 sequences at 131072 context, llama3 rope scaling
  5 phi4_gemma2_mixed        8 prefill chunks x 1024 + 120 decode tokens, Hq=24, Hkv=8, d=128,
                             96 rotated dims, longrope, soft-cap 50, a windowed and a full layer

Each builder takes ``scale``: "full" is the workload itself; "small" keeps its structure (several tiles,
ragged tails, windows that bind, longrope on both sides of its switch) at sizes the fp64 oracle finishes
in seconds; "profile" (decode and mixed workloads) keeps the full head shapes with fewer sequences or
shorter contexts, so that the caches stay within a few GB for profiler captures. Tensor draws come from a ``torch.Generator`` seeded with 1000 + workload number, in a fixed
order (q, k, v, norm weights, cache K, cache V); context lengths, chunk starts and row permutations come
from a second CPU generator seeded with 2000 + workload number. Full-size caches are drawn on the device
from a generator of their own, so that no multi-GB tensor is staged on the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NAMES = {
    1: "tiny_prefill_fp32",
    2: "qwen3_8b_prefill",
    3: "mistral_swa_decode",
    4: "llama31_8b_long_decode",
    5: "phi4_gemma2_mixed",
}
NUMBERS = {v: k for k, v in NAMES.items()}


@dataclass
class LayerCall:
    """Everything one layer's attention step reads.

    Tokens are laid out prefill-first: tokens [0, n_prefill) belong to the prefill chunks (sequence b owns
    q_start[b] .. q_start[b+1]-1 at positions first_pos[b] + i), tokens [n_prefill, N) are decode tokens,
    one per decode sequence. Caches are [R, Hkv, M, d]; slot index = position.
    """
    head_dim: int
    num_attention_heads: int
    num_key_value_heads: int
    partial_rotary_factor: float
    rope_theta: float
    rope_scaling: dict | None
    max_position_embeddings: int
    dtype: torch.dtype
    window: int = 0
    softcap: float = 0.0
    eps: float = 1e-6
    q_norm_w: torch.Tensor | None = None        # fp32 [d] or None
    k_norm_w: torch.Tensor | None = None
    sinks: torch.Tensor | None = None           # fp32 [Hq] learned sink logits or None
    # new tokens
    q: torch.Tensor = None                       # [N, Hq, d]
    k: torch.Tensor = None                       # [N, Hkv, d]
    v: torch.Tensor = None                       # [N, Hkv, d]
    tok_rows: torch.Tensor = None                # int32 [N]
    tok_pos: torch.Tensor = None                 # int32 [N]
    tok_seq_len: torch.Tensor = None             # int32 [N] total length of the token's sequence
    # prefill part
    n_prefill: int = 0
    q_start: torch.Tensor = None                 # int32 [Sp+1]
    pf_rows: torch.Tensor = None                 # int32 [Sp]
    pf_first_pos: torch.Tensor = None            # int32 [Sp]
    max_q_len: int = 0
    # decode part
    dec_rows: torch.Tensor = None                # int32 [Sd]
    dec_pos: torch.Tensor = None                 # int32 [Sd]
    # caches
    k_cache: torch.Tensor = None                 # [R, Hkv, M, d]
    v_cache: torch.Tensor = None
    meta: dict = field(default_factory=dict)

    @property
    def n_tokens(self):
        return int(self.q.shape[0])

    @property
    def num_rows(self):
        return int(self.k_cache.shape[0])

    @property
    def max_len(self):
        return int(self.k_cache.shape[2])

    @property
    def n_decode(self):
        return self.n_tokens - self.n_prefill

    def to(self, device):
        out = LayerCall(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in self.__dataclass_fields__:
            val = getattr(self, k)
            if isinstance(val, torch.Tensor):
                setattr(out, k, val.to(device))
        out.meta = dict(self.meta)
        return out



# ------------------------------------------------------------------------------------------ MLA decode

DEEPSEEK_V3_YARN = {"type": "yarn", "factor": 40.0, "original_max_position_embeddings": 4096, "beta_fast": 32.0,
                    "beta_slow": 1.0, "mscale": 1.0, "mscale_all_dim": 1.0}


@dataclass
class MlaCall:
    """One MLA decode step: S sequences, one new token each (DeepSeek-V3 shapes: latent 512, rotary 64)."""
    num_heads: int
    qk_nope_head_dim: int            # the scale is (qk_nope + qk_rope)^-0.5 with YaRN's temperature
    qk_rope_head_dim: int
    rope_theta: float
    rope_scaling: dict | None
    max_position_embeddings: int
    q: torch.Tensor = None           # [S, H, 576] bf16: W_uk^T q_nope (512), then q_rope (64, adjacent pairs)
    latent: torch.Tensor = None      # [S, 512] bf16: the new token's latent c
    k_rope: torch.Tensor = None      # [S, 64] bf16: its rotary key (adjacent pairs)
    rows: torch.Tensor = None        # int32 [S]
    positions: torch.Tensor = None   # int32 [S]: the new token's position (it sees 0..p)
    seq_len: torch.Tensor = None     # int32 [S]: positions + 1
    cache: torch.Tensor = None       # [R, M, 576] bf16: rows [c, rotated k_rope] of earlier positions
    window: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def n_seqs(self):
        return int(self.q.shape[0])

    @property
    def num_rows(self):
        return int(self.cache.shape[0])

    @property
    def max_len(self):
        return int(self.cache.shape[1])

    def to(self, device):
        out = MlaCall(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in self.__dataclass_fields__:
            val = getattr(self, k)
            if isinstance(val, torch.Tensor):
                setattr(out, k, val.to(device))
        out.meta = dict(self.meta)
        return out


def deepseek_v3_mla_decode(scale="full", device="cpu", heads=128):
    """MLA decode with DeepSeek-V3's attention shapes: 128 query heads per latent row, rows of 512 + 64,
    YaRN (factor 40 over 4096), one new token for each of 64 sequences at contexts uniform in [2048, 32768]
    (rows permuted). Latents and rotary keys N(0,1); absorbed queries N(0, 0.5^2). Small: 5 sequences at
    contexts up to 700 (one first token, one at the 64-key tile boundary), 16 heads."""
    g = _gen(1006)
    g_len = _gen(2006)
    if scale == "full":
        S, lo, hi, M, H = 64, 2048, 32768, 32768, heads
        lens = torch.randint(lo, hi + 1, (S,), generator=g_len).tolist()
    else:
        S, M, H = 5, 700, 16
        lens = [1, 64, 65, 700, 333]
    rows = torch.randperm(S, generator=g_len).tolist()
    cache = torch.empty((S, M, 576), dtype=torch.bfloat16, device=device)
    gd = g if str(device) == "cpu" else _gen(1006 + 7919, device)
    for r in range(S):
        cache[r].copy_(torch.randn((M, 576), generator=gd, dtype=torch.float32, device=device))
    q = _randn(g, (S, H, 576), 0.5, torch.bfloat16)
    latent = _randn(g, (S, 512), 1.0, torch.bfloat16)
    k_rope = _randn(g, (S, 64), 1.0, torch.bfloat16)
    pos = [L - 1 for L in lens]
    return MlaCall(num_heads=H, qk_nope_head_dim=128, qk_rope_head_dim=64, rope_theta=1e4, rope_scaling=DEEPSEEK_V3_YARN,
                   max_position_embeddings=163840, q=q, latent=latent, k_rope=k_rope, rows=_i32(rows),
                   positions=_i32(pos), seq_len=_i32(lens), cache=cache,
                   meta={"description": f"DeepSeek-V3 MLA decode: {S} sequences, {H} heads per 576-wide latent row, "
                                        f"contexts {min(lens)}..{max(lens)}"}).to(device)


def paged_from_contiguous(k_cache, v_cache, block_size, seed=0, spare_blocks=0, unmap_before=None, unmap_from=None):
    """A paged pool holding the blocks of contiguous caches [R, Hkv, M, d] in a seeded random order.

    Returns (k_pool, v_pool, block_table): pools [n_blocks, Hkv, block_size, d] (n_blocks = R * ceil(M /
    block_size) + spare_blocks; spare blocks and the tail of a row's last block hold NaN) and an int32 table
    [R, ceil(M / block_size)]. unmap_before[r], if given, unmaps (-1, contents NaN) every block of row r that
    lies wholly before that position, as a pool that recycles out-of-window blocks leaves them; unmap_from[r]
    unmaps every block that starts at or after that position, as a pool that maps blocks only as a row
    grows leaves them."""
    R, hkv, M, d = k_cache.shape
    nb = (M + block_size - 1) // block_size
    n_blocks = R * nb + spare_blocks
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_blocks, generator=g)[:R * nb].reshape(R, nb)
    kp = torch.full((n_blocks, hkv, block_size, d), float("nan"), dtype=k_cache.dtype, device=k_cache.device)
    vp = torch.full_like(kp, float("nan"))
    pad = nb * block_size - M
    kc = torch.nn.functional.pad(k_cache, (0, 0, 0, pad), value=float("nan")) if pad else k_cache
    vc = torch.nn.functional.pad(v_cache, (0, 0, 0, pad), value=float("nan")) if pad else v_cache
    idx = perm.reshape(-1).to(k_cache.device)
    kp[idx] = kc.reshape(R, hkv, nb, block_size, d).transpose(1, 2).reshape(R * nb, hkv, block_size, d)
    vp[idx] = vc.reshape(R, hkv, nb, block_size, d).transpose(1, 2).reshape(R * nb, hkv, block_size, d)
    table = perm.clone().to(torch.int32)
    if unmap_before is not None or unmap_from is not None:
        for r in range(R):
            for b in range(nb):
                gone = unmap_before is not None and (b + 1) * block_size <= int(unmap_before[r])
                gone = gone or (unmap_from is not None and b * block_size >= int(unmap_from[r]))
                if gone:
                    kp[perm[r, b]] = float("nan")
                    vp[perm[r, b]] = float("nan")
                    table[r, b] = -1
    return kp, vp, table.to(k_cache.device)

@dataclass
class Workload:
    number: int
    name: str
    scale: str
    layers: list                                 # [LayerCall]

    @property
    def description(self):
        return self.layers[0].meta.get("description", self.name)


def _gen(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(g, shape, std=1.0, dtype=torch.float32, device="cpu"):
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _fill_cache(g, shape, dtype, device, chunk_rows=1):
    """A cache [R, Hkv, M, d] of N(0,1) values, drawn row by row to bound the fp32 staging buffer."""
    out = torch.empty(shape, dtype=dtype, device=device)
    for r in range(0, shape[0], chunk_rows):
        out[r:r + chunk_rows].copy_(torch.randn((min(chunk_rows, shape[0] - r),) + tuple(shape[1:]),
                                                generator=g, dtype=torch.float32, device=device))
    return out


def _i32(x, device="cpu"):
    return torch.as_tensor(x, dtype=torch.int32, device=device)


def _prefill_meta(chunk_lens, first_pos, rows):
    q_start = [0]
    for n in chunk_lens:
        q_start.append(q_start[-1] + int(n))
    tok_rows, tok_pos, tok_len = [], [], []
    for n, p0, r in zip(chunk_lens, first_pos, rows):
        tok_rows += [int(r)] * int(n)
        tok_pos += list(range(int(p0), int(p0) + int(n)))
        tok_len += [int(p0) + int(n)] * int(n)
    return q_start, tok_rows, tok_pos, tok_len


# --------------------------------------------------------------------------------------------------

def tiny_prefill_fp32(scale="full", device="cpu"):
    """Workload 1: B=1, 128 tokens, Hq=4, Hkv=2, d=64, fp32, plain RoPE theta 1e4, positions 0..127."""
    g = _gen(1001)
    T, hq, hkv, d = 128, 4, 2, 64
    q = _randn(g, (T, hq, d))
    k = _randn(g, (T, hkv, d))
    v = _randn(g, (T, hkv, d))
    kc = torch.zeros((1, hkv, T, d), dtype=torch.float32)
    vc = torch.zeros_like(kc)
    q_start, tr, tp, tl = _prefill_meta([T], [0], [0])
    call = LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, partial_rotary_factor=1.0,
                     rope_theta=1e4, rope_scaling=None, max_position_embeddings=4096, dtype=torch.float32,
                     q=q, k=k, v=v, tok_rows=_i32(tr), tok_pos=_i32(tp), tok_seq_len=_i32(tl),
                     n_prefill=T, q_start=_i32(q_start), pf_rows=_i32([0]), pf_first_pos=_i32([0]), max_q_len=T,
                     dec_rows=_i32([]), dec_pos=_i32([]), k_cache=kc, v_cache=vc,
                     meta={"description": "tiny fp32 prefill, B=1 x 128, Hq=4, Hkv=2, d=64"})
    return Workload(1, NAMES[1], scale, [call.to(device)])


def qwen3_8b_prefill(scale="full", device="cpu"):
    """Workload 2: B=4 x 2048 tokens (small: 3 chunks of 200/333/77), Hq=32, Hkv=8, d=128, bf16, q/k RMSNorm
    eps 1e-6 with weights 1 + N(0, 0.02), theta 1e6, activations N(0,1)/sqrt(128), cache written at 0.."""
    g = _gen(1002)
    hq, hkv, d = 32, 8, 128
    if scale == "full":
        lens = [2048] * 4
        hq_, hkv_ = hq, hkv
    else:
        lens = [200, 333, 77]
        hq_, hkv_ = 8, 2
    n = sum(lens)
    std = 1.0 / math.sqrt(d)
    q = _randn(g, (n, hq_, d), std, torch.bfloat16)
    k = _randn(g, (n, hkv_, d), std, torch.bfloat16)
    v = _randn(g, (n, hkv_, d), std, torch.bfloat16)
    wq = 1.0 + _randn(g, (d,), 0.02)
    wk = 1.0 + _randn(g, (d,), 0.02)
    R, M = len(lens), max(lens)
    kc = torch.zeros((R, hkv_, M, d), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    rows = list(range(R))
    q_start, tr, tp, tl = _prefill_meta(lens, [0] * R, rows)
    call = LayerCall(head_dim=d, num_attention_heads=hq_, num_key_value_heads=hkv_, partial_rotary_factor=1.0,
                     rope_theta=1e6, rope_scaling=None, max_position_embeddings=40960, dtype=torch.bfloat16,
                     eps=1e-6, q_norm_w=wq, k_norm_w=wk,
                     q=q, k=k, v=v, tok_rows=_i32(tr), tok_pos=_i32(tp), tok_seq_len=_i32(tl),
                     n_prefill=n, q_start=_i32(q_start), pf_rows=_i32(rows), pf_first_pos=_i32([0] * R),
                     max_q_len=max(lens), dec_rows=_i32([]), dec_pos=_i32([]), k_cache=kc, v_cache=vc,
                     meta={"description": f"Qwen3-8B-shaped prefill, {len(lens)} x {lens}, Hq={hq_}, Hkv={hkv_}, d=128"})
    call = call.to(device)
    return Workload(2, NAMES[2], scale, [call])


def _decode_call(g, device, lens, hq, hkv, d, R, M, rows, dtype, q_std, **kw):
    """Decode tokens at positions lens-1; the cache rows hold N(0,1) keys/values (drawn on `device`)."""
    S = len(lens)
    q = _randn(g, (S, hq, d), q_std, dtype)
    k = _randn(g, (S, hkv, d), 1.0, dtype)
    v = _randn(g, (S, hkv, d), 1.0, dtype)
    gd = g if str(device) == "cpu" else _gen(g.initial_seed() + 7919, device)
    kc = _fill_cache(gd, (R, hkv, M, d), dtype, device)
    vc = _fill_cache(gd, (R, hkv, M, d), dtype, device)
    pos = [int(L) - 1 for L in lens]
    call = LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, dtype=dtype,
                     q=q, k=k, v=v, tok_rows=_i32(rows), tok_pos=_i32(pos), tok_seq_len=_i32(lens),
                     n_prefill=0, q_start=_i32([0]), pf_rows=_i32([]), pf_first_pos=_i32([]), max_q_len=0,
                     dec_rows=_i32(rows), dec_pos=_i32(pos), k_cache=kc, v_cache=vc, **kw)
    return call


def mistral_swa_decode(scale="full", device="cpu"):
    """Workload 3: 64 sequences, contexts uniform in [1024, 32768] (small: 12 in [40, 2000], window 300),
    Hq=32, Hkv=8, d=128, sliding window 4096, theta 1e6, rows a random permutation."""
    g = _gen(1003)
    if scale == "full":
        S, lo, hi, w, hq, hkv, M = 64, 1024, 32768, 4096, 32, 8, 32768
    elif scale == "profile":
        S, lo, hi, w, hq, hkv, M = 16, 1024, 32768, 4096, 32, 8, 32768
    else:
        S, lo, hi, w, hq, hkv, M = 12, 40, 2000, 300, 8, 2, 2000
    d = 128
    g_len = _gen(2003)
    lens = torch.randint(lo, hi + 1, (S,), generator=g_len).tolist()
    rows = torch.randperm(S, generator=g_len).tolist()
    call = _decode_call(g, device, lens, hq, hkv, d, S, M, rows, torch.bfloat16, 1.0 / math.sqrt(d),
                        partial_rotary_factor=1.0, rope_theta=1e6, rope_scaling=None,
                        max_position_embeddings=32768, window=w,
                        meta={"description": f"Mistral-style sliding-window decode, {S} seqs, ctx U[{lo},{hi}], w={w}"})
    return Workload(3, NAMES[3], scale, [call.to(device)])


def llama31_8b_long_decode(scale="full", device="cpu"):
    """Workload 4: 16 sequences at context 131072 (small: 4 at 3000, 2500, 700, 1), Hq=32, Hkv=8, d=128,
    full causal, theta 5e5 with llama3 scaling (factor 8, low 1, high 4, original 8192)."""
    g = _gen(1004)
    d = 128
    if scale == "full":
        lens, hq, hkv, M = [131072] * 16, 32, 8, 131072
    elif scale == "profile":
        lens, hq, hkv, M = [16384] * 16, 32, 8, 16384
    else:
        lens, hq, hkv, M = [3000, 2500, 700, 1], 8, 2, 3000
    S = len(lens)
    rows = list(range(S))
    scaling = {"rope_type": "llama3", "factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
               "original_max_position_embeddings": 8192}
    call = _decode_call(g, device, lens, hq, hkv, d, S, M, rows, torch.bfloat16, 1.0 / math.sqrt(d),
                        partial_rotary_factor=1.0, rope_theta=5e5, rope_scaling=scaling,
                        max_position_embeddings=131072,
                        meta={"description": f"Llama-3.1-8B-shaped decode, {S} seqs at {max(lens)} context, llama3 scaling"})
    return Workload(4, NAMES[4], scale, [call.to(device)])


def phi4_longrope_scaling(rot_half=48):
    """Synthetic LongRoPE tables: short ascending in [1.0, 1.2], long ascending in [1.0, 40.0]."""
    short = torch.linspace(1.0, 1.2, rot_half, dtype=torch.float64).tolist()
    long_ = torch.linspace(1.0, 40.0, rot_half, dtype=torch.float64).tolist()
    return {"rope_type": "longrope", "short_factor": short, "long_factor": long_,
            "original_max_position_embeddings": 4096}


def phi4_gemma2_mixed(scale="full", device="cpu", q_mult=1.0):
    """Workload 5: a windowed layer (w=4096) and a full layer over one mixed batch: 8 prefill chunks of 1024
    tokens at starts uniform in [0, 64512] plus 120 decode tokens at contexts uniform in [512, 65536];
    Hq=24, Hkv=8, d=128, 96 rotated dims, longrope (original 4096, max 131072), soft-cap 50, theta 1e4,
    Q/K/V N(0,1). Rows: chunks 0..7, decode tokens a permutation of 8..127. q_mult > 1 scales q so that the
    cap binds. Small: 3 chunks of 100 + 9 decode tokens, contexts to 6000, window 512, Hq=6, Hkv=2."""
    g = _gen(1005)
    d = 128
    if scale == "full":
        n_chunks, chunk, n_dec, dlo, dhi, pmax, w, hq, hkv = 8, 1024, 120, 512, 65536, 64512, 4096, 24, 8
        M = 65536
    elif scale == "profile":
        n_chunks, chunk, n_dec, dlo, dhi, pmax, w, hq, hkv = 6, 1024, 8, 512, 24576, 23552, 4096, 24, 8
        M = 24576
    else:
        n_chunks, chunk, n_dec, dlo, dhi, pmax, w, hq, hkv = 3, 100, 9, 50, 6000, 5800, 512, 6, 2
        M = 6000
    R = n_chunks + n_dec
    g_len = _gen(2005)
    starts = torch.randint(0, pmax + 1, (n_chunks,), generator=g_len).tolist()
    if scale != "full":
        starts[0] = 0                    # one chunk from position 0
        starts[1] = 4000                 # one chunk that straddles the longrope switch (4096)
    dec_lens = torch.randint(dlo, dhi + 1, (n_dec,), generator=g_len).tolist()
    if scale != "full":
        dec_lens[0] = 4096               # exactly at the switch: short table
        dec_lens[1] = 4097               # one past: long table
        dec_lens[2] = 1                  # a first token
    dec_rows = (torch.randperm(n_dec, generator=g_len) + n_chunks).tolist()
    scaling = phi4_longrope_scaling(48)
    layers = []
    for li, window in enumerate((w, 0)):
        lens = [chunk] * n_chunks
        q_start, tr, tp, tl = _prefill_meta(lens, starts, list(range(n_chunks)))
        n = n_chunks * chunk + n_dec
        q = _randn(g, (n, hq, d), q_mult, torch.bfloat16)
        k = _randn(g, (n, hkv, d), 1.0, torch.bfloat16)
        v = _randn(g, (n, hkv, d), 1.0, torch.bfloat16)
        gd = g if str(device) == "cpu" else _gen(1005 + 7919 + li, device)
        kc = _fill_cache(gd, (R, hkv, M, d), torch.bfloat16, device)
        vc = _fill_cache(gd, (R, hkv, M, d), torch.bfloat16, device)
        dec_pos = [L - 1 for L in dec_lens]
        call = LayerCall(head_dim=d, num_attention_heads=hq, num_key_value_heads=hkv, partial_rotary_factor=0.75,
                         rope_theta=1e4, rope_scaling=scaling, max_position_embeddings=131072,
                         dtype=torch.bfloat16, window=window, softcap=50.0,
                         q=q, k=k, v=v,
                         tok_rows=_i32(tr + dec_rows), tok_pos=_i32(tp + dec_pos), tok_seq_len=_i32(tl + dec_lens),
                         n_prefill=n_chunks * chunk, q_start=_i32(q_start), pf_rows=_i32(list(range(n_chunks))),
                         pf_first_pos=_i32(starts), max_q_len=chunk,
                         dec_rows=_i32(dec_rows), dec_pos=_i32(dec_pos), k_cache=kc, v_cache=vc,
                         meta={"description": f"Phi-4-mini/Gemma-2-style layer {li} ({'window ' + str(window) if window else 'full'}), "
                                              f"{n_chunks} x {chunk} prefill + {n_dec} decode"})
        layers.append(call.to(device))
    return Workload(5, NAMES[5], scale, layers)


BUILDERS = {1: tiny_prefill_fp32, 2: qwen3_8b_prefill, 3: mistral_swa_decode, 4: llama31_8b_long_decode,
            5: phi4_gemma2_mixed}


def make(workload, scale="full", device="cpu", **kw):
    """Build workload `workload` (number or name)."""
    num = workload if isinstance(workload, int) else NUMBERS[workload]
    return BUILDERS[num](scale=scale, device=device, **kw)


def subset(call: LayerCall, chunks, decode_idx, device="cpu", kv_heads=None, kv_first=0) -> LayerCall:
    """A LayerCall holding only prefill chunks `chunks` and decode tokens `decode_idx` of `call`, with the
    cache rows they use (renumbered 0..k-1) copied to `device`; with `kv_heads`, only KV heads
    kv_first .. kv_first + kv_heads - 1 and their query-head groups. Bookkeeping only: used to size bounded
    samples of a full workload for the CPU oracle."""
    chunks = list(chunks)
    hkv = call.num_key_value_heads if kv_heads is None else int(kv_heads)
    grp = call.num_attention_heads // call.num_key_value_heads
    hq = hkv * grp
    g0, g1 = kv_first, kv_first + hkv
    q0, q1 = g0 * grp, g1 * grp
    decode_idx = list(decode_idx)
    qs = call.q_start.cpu().tolist()
    pf_rows = call.pf_rows.cpu().tolist()
    pf_fp = call.pf_first_pos.cpu().tolist()
    dec_rows = call.dec_rows.cpu().tolist()
    dec_pos = call.dec_pos.cpu().tolist()
    rows_used = [pf_rows[b] for b in chunks] + [dec_rows[i] for i in decode_idx]
    remap = {r: j for j, r in enumerate(dict.fromkeys(rows_used))}
    tok = []
    lens = []
    for b in chunks:
        tok += list(range(qs[b], qs[b + 1]))
        lens.append(qs[b + 1] - qs[b])
    n_pf = len(tok)
    tok += [call.n_prefill + i for i in decode_idx]
    idx = torch.as_tensor(tok, dtype=torch.long)
    q_start, tr, tp, tl = _prefill_meta(lens, [pf_fp[b] for b in chunks], [remap[pf_rows[b]] for b in chunks])
    d_rows = [remap[dec_rows[i]] for i in decode_idx]
    d_pos = [dec_pos[i] for i in decode_idx]
    d_len = [p + 1 for p in d_pos]
    ridx = torch.as_tensor(list(remap.keys()), dtype=torch.long, device=call.k_cache.device)
    fields = {k: getattr(call, k) for k in call.__dataclass_fields__}
    fields.update(
        num_attention_heads=hq, num_key_value_heads=hkv,
        q=call.q[idx.to(call.q.device), q0:q1].to(device), k=call.k[idx.to(call.k.device), g0:g1].to(device),
        v=call.v[idx.to(call.v.device), g0:g1].to(device),
        tok_rows=_i32(tr + d_rows, device), tok_pos=_i32(tp + d_pos, device), tok_seq_len=_i32(tl + d_len, device),
        n_prefill=n_pf, q_start=_i32(q_start, device), pf_rows=_i32([remap[pf_rows[b]] for b in chunks], device),
        pf_first_pos=_i32([pf_fp[b] for b in chunks], device), max_q_len=max(lens) if lens else 0,
        dec_rows=_i32(d_rows, device), dec_pos=_i32(d_pos, device),
        k_cache=call.k_cache[ridx, g0:g1].to(device), v_cache=call.v_cache[ridx, g0:g1].to(device),
        sinks=call.sinks[q0:q1].to(device) if call.sinks is not None else None,
        q_norm_w=call.q_norm_w.to(device) if call.q_norm_w is not None else None,
        k_norm_w=call.k_norm_w.to(device) if call.k_norm_w is not None else None,
        meta=dict(call.meta))
    return LayerCall(**fields)
