// RoPE tables and the fused q/k RMSNorm + RoPE + KV-cache write.
//
// Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention": rope_tables
// (section "Scaled RoPE") and the part of DecoderAttention.forward from q_norm/k_norm through
// cache.update; page "MoE, optimisers, decoding -- every line, every shape", §3.2 RMSNorm, §3.3 KVCache
// and §4 Rotary for the norm, the cache write and the split-half rotation.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {

// ---------------------------------------------------------------------------------------------- tables

// inv / (2 pi) as a fixed-point fraction of 2^64 (inv < 2 pi for every RoPE pair, so the value is < 1).
// fp64 carries 53 bits of it, the same precision an fp64 angle product would have.
static unsigned long long turn_fixed(double inv) {
  const double f = inv / 6.283185307179586476925286766559;   // turns per position
  const double hi = std::floor(std::ldexp(f, 32));
  const double lo = std::floor(std::ldexp(std::ldexp(f, 32) - hi, 32));
  return (static_cast<unsigned long long>(hi) << 32) | static_cast<unsigned long long>(lo);
}

RopeTurns rope_turns(const RopeFreqs& f) {
  RopeTurns t;
  t.half = f.half;
  t.switch_len = f.switch_len;
  t.use_seq_len = f.use_seq_len;
  t.af = static_cast<float>(f.af);
  for (int i = 0; i < kMaxRotHalf; ++i) {
    t.turn_short[i] = i < f.half ? turn_fixed(f.inv_short[i]) : 0ull;
    t.turn_long[i] = i < f.half ? turn_fixed(f.inv_long[i]) : 0ull;
  }
  return t;
}

// One thread per (token, four consecutive pairs): the token's position (and sequence length) is loaded once
// for the four. p * turns (mod 2^64) is the angle's fraction of a full turn, exactly up to the table's 53
// significant bits; its top 32 bits, read as a signed fraction x in [-1, 1), give the angle pi * x in
// [-pi, pi), whose sine and cosine sincospif takes in fp32. At p ~ 131071 an fp32 product p * inv would be
// off by up to 4e-3 rad; this stays within ~2e-7.
constexpr int kRopePairs = 4;
__global__ void rope_tables_kernel(const __grid_constant__ RopeTurns f, const int32_t* __restrict__ positions,
                                   const int32_t* __restrict__ seq_len, int n, float* __restrict__ cos_out,
                                   float* __restrict__ sin_out, int* err) {
  const int groups = (f.half + kRopePairs - 1) / kRopePairs;   // pair groups per token
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n) * groups) return;
  const int t = static_cast<int>(idx / groups);
  const int i0 = static_cast<int>(idx - static_cast<long long>(t) * groups) * kRopePairs;
  pdl_wait();   // inputs written by the stream's previous kernel are visible
  const int p = positions[t];
  const bool use_long = f.use_seq_len && seq_len[t] > f.switch_len;
  float c[kRopePairs], s[kRopePairs];
#pragma unroll
  for (int j = 0; j < kRopePairs; ++j) {
    const int i = i0 + j;
    const unsigned long long turn = i < f.half ? (use_long ? f.turn_long[i] : f.turn_short[i]) : 0ull;
    const unsigned long long frac = static_cast<unsigned long long>(p) * turn;     // mod 2^64
    const int top = static_cast<int>(static_cast<unsigned int>(frac >> 32));      // signed fraction of 2^31
    const float x = static_cast<float>(top) * 4.656612873077393e-10f;             // top / 2^31
    sincospif(x, &s[j], &c[j]);
    c[j] *= f.af;
    s[j] *= f.af;
  }
  if (p < 0) {
    if (i0 == 0) set_error(err, kErrIndex);
#pragma unroll
    for (int j = 0; j < kRopePairs; ++j) c[j] = s[j] = 0.f;
  }
  const long long o = static_cast<long long>(t) * f.half + i0;
  if (f.half % kRopePairs == 0) {   // rows of 16-byte multiples: vector stores
    *reinterpret_cast<float4*>(cos_out + o) = make_float4(c[0], c[1], c[2], c[3]);
    *reinterpret_cast<float4*>(sin_out + o) = make_float4(s[0], s[1], s[2], s[3]);
  } else {
#pragma unroll
    for (int j = 0; j < kRopePairs; ++j) {
      if (i0 + j < f.half) {
        cos_out[o + j] = c[j];
        sin_out[o + j] = s[j];
      }
    }
  }
}

cudaError_t launch_rope_tables(const RopeFreqs& f, const int32_t* positions, const int32_t* seq_len, int n,
                               float* cos, float* sin, int* err, cudaStream_t stream) {
  const long long total = static_cast<long long>(n) * ((f.half + kRopePairs - 1) / kRopePairs);
  if (total == 0) return cudaSuccess;
  const RopeTurns turns = rope_turns(f);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  return launch_dependent(rope_tables_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, turns,
                          positions, seq_len, n, cos, sin, err);
}

// ---------------------------------------------------------------------------------------------- cache update

template <typename T>
struct Vec16;
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f2 = __bfloat1622float2(h[j]);
      x[2 * j] = f2.x;
      x[2 * j + 1] = f2.y;
    }
  }
  __device__ static void store(void* p, const float (&x)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float (&x)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  }
  __device__ static void store(void* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};

// One warp per token. Lane l owns the 16-byte piece sub = l % TPV (VEC consecutive elements) of a head
// vector, TPV = d / VEC lanes per vector, HPW = 32 / TPV vectors per warp at a time; the warp walks the
// token's Hq query heads then its Hkv key heads. A key head also copies the token's value vector into the
// V cache (bit for bit). A lane's cos/sin entries and norm weights depend only on its piece, so they are
// loaded once per token.
// SHFL: r/2 is a multiple of VEC, so the rotation partner of a lane's piece (elements i +- r/2) is another
// lane's whole piece: it comes by warp shuffle. Otherwise the normalised vector is staged in shared memory.
template <typename T, int D, bool SHFL>
__global__ void __launch_bounds__(256) kv_update_kernel(const KvUpdateArgs a) {
  using V = Vec16<T>;
  constexpr int VEC = V::N;
  constexpr int TPV = D / VEC;            // lanes per vector (8..32)
  constexpr int HPW = 32 / TPV;           // vectors per warp per step
  constexpr int WPB = 8;                  // warps per block
  __shared__ float stage[SHFL ? 1 : WPB][SHFL ? 1 : HPW][SHFL ? 1 : D];

  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  // a.wpt warps share a token when tokens are few (decode), each taking every wpt-th group of heads
  const long long gw = static_cast<long long>(blockIdx.x) * WPB + wib;
  const int t = static_cast<int>(gw / a.wpt);
  const int part = static_cast<int>(gw - static_cast<long long>(t) * a.wpt);
  if (t >= a.n) return;                   // whole warps leave together
  pdl_wait();                             // inputs written by the stream's previous kernel are visible
  const int sub = lane % TPV;
  const int slot = lane / TPV;
  const int e0 = sub * VEC;
  const int half = a.rot >> 1;
  const int heads = a.hq + a.hkv;

  // per-token, per-piece data: cos/sin of the piece's pairs, norm weights, the token's cache slot
  float c[VEC], sv[VEC], wq[VEC], wk[VEC];
  const int hc = half / VEC;               // pieces per half (SHFL path)
  const bool lower = SHFL && sub < hc, upper = SHFL && sub >= hc && sub < 2 * hc;
  if (SHFL && (lower || upper)) {
    const int ci = (lower ? sub : sub - hc) * VEC;
    const float* cs = a.cos + static_cast<long long>(t) * half + ci;
    const float* sn = a.sin + static_cast<long long>(t) * half + ci;
#pragma unroll
    for (int j = 0; j < VEC; j += 4) {
      const float4 c4 = *reinterpret_cast<const float4*>(cs + j);
      const float4 s4 = *reinterpret_cast<const float4*>(sn + j);
      c[j] = c4.x; c[j + 1] = c4.y; c[j + 2] = c4.z; c[j + 3] = c4.w;
      sv[j] = s4.x; sv[j + 1] = s4.y; sv[j + 2] = s4.z; sv[j + 3] = s4.w;
    }
  }
  const bool norm = a.q_norm_w != nullptr;
  if (norm) {
#pragma unroll
    for (int j = 0; j < VEC; j += 4) {
      const float4 q4 = *reinterpret_cast<const float4*>(a.q_norm_w + e0 + j);
      const float4 k4 = *reinterpret_cast<const float4*>(a.k_norm_w + e0 + j);
      wq[j] = q4.x; wq[j + 1] = q4.y; wq[j + 2] = q4.z; wq[j + 3] = q4.w;
      wk[j] = k4.x; wk[j + 1] = k4.y; wk[j + 2] = k4.z; wk[j + 3] = k4.w;
    }
  }
  const KvLayout kvl = kv_layout(a);
  const long long cslot = kv_slot(kvl, a.rows[t], a.positions[t]);
  const bool slot_ok = cslot >= 0;
  if (!slot_ok && lane == 0) set_error(a.err, kErrIndex);
  const long long slot_base = slot_ok ? cslot * D : 0;
  const long long head_step = kv_head_stride(kvl) * D;

  // U heads per lane are loaded before any is processed: enough loads in flight to cover HBM latency
  constexpr int U = 4;
  const int steps = (heads + HPW - 1) / HPW;
  for (int it0 = part; it0 < steps; it0 += U * a.wpt) {
    uint4 xr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int hh = (it0 + u * a.wpt) * HPW + slot;
      xr[u] = make_uint4(0, 0, 0, 0);
      vr[u] = make_uint4(0, 0, 0, 0);
      if (hh < heads) {
        const bool q_head = hh < a.hq;
        const T* src = q_head ? static_cast<const T*>(a.q) + (static_cast<long long>(t) * a.hq + hh) * D
                              : static_cast<const T*>(a.k) + (static_cast<long long>(t) * a.hkv + (hh - a.hq)) * D;
        xr[u] = *reinterpret_cast<const uint4*>(src + e0);
        if (!q_head)
          vr[u] = *reinterpret_cast<const uint4*>(static_cast<const T*>(a.v) +
                                                  (static_cast<long long>(t) * a.hkv + (hh - a.hq)) * D + e0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int it = it0 + u * a.wpt;
      const int hh = it * HPW + slot;
      const bool live = hh < heads;
      const bool is_q = hh < a.hq;
      const int g = hh - a.hq;
      float x[VEC];
      V::load(&xr[u], x);
      const uint4 vv = vr[u];
      // RMSNorm over the head: x / sqrt(mean(x^2) + eps) * w
      if (norm) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
        for (int off = TPV / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off, TPV);
        const float rs = rsqrtf(ss * (1.0f / D) + a.eps);
#pragma unroll
        for (int j = 0; j < VEC; ++j) x[j] = x[j] * rs * (is_q ? wq[j] : wk[j]);
      }
      // split-half rotation of the first `rot` dims: x'_i = x_i c - x_{i+h} s, x'_{i+h} = x_{i+h} c + x_i s
      float y[VEC];
      if (SHFL) {
        const int psub = lower ? sub + hc : (upper ? sub - hc : sub);
        const int src_lane = slot * TPV + psub;
        float px[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) px[j] = __shfl_sync(0xffffffffu, x[j], src_lane);
        if (lower || upper) {
          const float sgn = lower ? -1.f : 1.f;
#pragma unroll
          for (int j = 0; j < VEC; ++j) y[j] = fmaf(sgn * px[j], sv[j], x[j] * c[j]);
        } else {
#pragma unroll
          for (int j = 0; j < VEC; ++j) y[j] = x[j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) stage[wib][slot][e0 + j] = x[j];
        __syncwarp();
        const float* cs = a.cos + static_cast<long long>(t) * half;
        const float* sn = a.sin + static_cast<long long>(t) * half;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          const int e = e0 + j;
          if (e < half) {
            y[j] = x[j] * cs[e] - stage[wib][slot][e + half] * sn[e];
          } else if (e < a.rot) {
            y[j] = x[j] * cs[e - half] + stage[wib][slot][e - half] * sn[e - half];
          } else {
            y[j] = x[j];
          }
        }
        __syncwarp();
      }
      if (!live) continue;
      if (is_q) {
        V::store(static_cast<T*>(a.q_rot) + (static_cast<long long>(t) * a.hq + hh) * D + e0, y);
      } else if (slot_ok) {
        const long long off = slot_base + g * head_step + e0;
        V::store(static_cast<T*>(a.k_cache) + off, y);
        *reinterpret_cast<uint4*>(static_cast<T*>(a.v_cache) + off) = vv;
      }
    }
  }
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Bulk-copy form (SHFL layouts with cos/sin rows a multiple of 16 bytes). A block walks tokens blockIdx.x,
// blockIdx.x + gridDim.x, ... through KB_STAGES shared-memory stages. Per token one thread copies the
// token's q, k and v rows and its cos/sin rows into a stage with cp.async.bulk (so the loads in flight do not
// depend on registers); warps 0-7 normalise and rotate the q and k heads in place (same lane layout as
// above); the same thread then stores the q row to q_rot and each K and V head to its cache slot with bulk
// copies (V never passes through registers) and refills the stage once the stores have read it.
constexpr int KB_STAGES = 4;
constexpr int KB_THREADS = 288;           // 8 computing warps + 1 copy warp
constexpr int KB_META = 64;               // tokens whose row / position a fused block reads ahead
struct KbLayout {                         // byte offsets within a stage
  int k, v, cos, sin, hdr, bytes;         // q at 0; hdr: the token's cache slot (8 bytes, -1: none)
};
static KbLayout kb_layout(int hq, int hkv, int d, int half, int es) {
  KbLayout L;
  L.k = hq * d * es;
  L.v = L.k + hkv * d * es;
  L.cos = L.v + hkv * d * es;
  L.sin = L.cos + half * 4;
  L.hdr = L.sin + half * 4;
  L.bytes = (L.hdr + 16 + 127) / 128 * 128;
  return L;
}

// FUSED: no cos/sin tables; per token the computing threads form its cos/sin (one rotary pair each) in the
// stage with the arithmetic of rope_tables_kernel, so the results are the same bits; bf16 with d = 128 only.
// Residency: the fused form fits 56 registers without spills, so four blocks share an SM (their stages,
// 4 x 51 KB on the Qwen3-8B shape, fit too); the table forms keep three (the bf16 d = 64 one spills at 56).
template <typename T, int D, bool FUSED>
__global__ void __launch_bounds__(KB_THREADS, FUSED ? 4 : 3) kv_update_bulk_kernel(const KvUpdateArgs a, const KbLayout L,
                                                                   const __grid_constant__ RopeTurns f) {
  using V = Vec16<T>;
  constexpr int VEC = V::N;
  constexpr int TPV = D / VEC;
  constexpr int HPW = 32 / TPV;
  extern __shared__ __align__(128) uint8_t kb_smem[];
  __shared__ uint64_t bars[2 * KB_STAGES];   // full[s] (copy + bytes), done[s] (256 computing threads)
  __shared__ int meta_row[FUSED ? KB_META : 1], meta_pos[FUSED ? KB_META : 1], meta_len[FUSED ? KB_META : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = a.rot >> 1;
  const int heads = a.hq + a.hkv;
  const int n_mine = a.n > static_cast<int>(blockIdx.x) ? (a.n - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const uint32_t sbase = smem_u32(kb_smem);
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto done = [&](int s) { return smem_u32(&bars[KB_STAGES + s]); };
  if (threadIdx.x == 0) {
    for (int s = 0; s < KB_STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(done(s), 256);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();   // inputs written by the stream's previous kernel are visible
  const int es = static_cast<int>(sizeof(T));
  const uint32_t in_bytes = static_cast<uint32_t>(FUSED ? L.cos : L.hdr);   // q, k, v (, cos, sin)

  if (warp == 8) {
    if (lane != 0) return;
    // ------------------------------------------------------------------ copies in and out
    auto issue = [&](int kk) {
      const int t = blockIdx.x + kk * gridDim.x;
      const int s = kk % KB_STAGES;
      const uint32_t st = sbase + s * L.bytes;
      mbar_arrive_expect_tx(full(s), in_bytes);
      bulk_load(st, static_cast<const T*>(a.q) + static_cast<long long>(t) * a.hq * D, a.hq * D * es, full(s));
      bulk_load(st + L.k, static_cast<const T*>(a.k) + static_cast<long long>(t) * a.hkv * D, a.hkv * D * es, full(s));
      bulk_load(st + L.v, static_cast<const T*>(a.v) + static_cast<long long>(t) * a.hkv * D, a.hkv * D * es, full(s));
      if (!FUSED) {
        bulk_load(st + L.cos, a.cos + static_cast<long long>(t) * half, half * 4, full(s));
        bulk_load(st + L.sin, a.sin + static_cast<long long>(t) * half, half * 4, full(s));
      }
    };
    int issued = 0;
    for (; issued < n_mine && issued < KB_STAGES; ++issued) issue(issued);
    for (int kk = 0; kk < n_mine; ++kk) {
      const int t = blockIdx.x + kk * gridDim.x;
      const int s = kk % KB_STAGES;
      const uint32_t st = sbase + s * L.bytes;
      if (!mbar_wait(done(s), (kk / KB_STAGES) & 1, a.err)) {
        // gave up (the error word is set): let the loads already issued for stages kk.. land before exiting
        for (int j = kk; j < issued; ++j) mbar_wait(full(j % KB_STAGES), (j / KB_STAGES) & 1, a.err);
        break;
      }
      const long long slot = *reinterpret_cast<const long long*>(kb_smem + s * L.bytes + L.hdr);
      bulk_store(static_cast<T*>(a.q_rot) + static_cast<long long>(t) * a.hq * D, st, a.hq * D * es);
      if (slot >= 0) {
        for (int g = 0; g < a.hkv; ++g) {
          const long long off = (slot + g * kv_head_stride(kv_layout(a))) * D;
          bulk_store(static_cast<T*>(a.k_cache) + off, st + L.k + g * D * es, D * es);
          bulk_store(static_cast<T*>(a.v_cache) + off, st + L.v + g * D * es, D * es);
        }
      }
      bulk_commit();
      if (kk + KB_STAGES < n_mine) {
        bulk_wait_read();   // the stage is refilled only after its stores have read it
        issue(kk + KB_STAGES);
        issued = kk + KB_STAGES + 1;
      }
    }
    bulk_wait_all();
    return;
  }

  // -------------------------------------------------------------------- normalise and rotate (warps 0-7)
  const bool norm = a.q_norm_w != nullptr;
  if constexpr (std::is_same_v<T, __nv_bfloat16> && D == 128) {
    // Two heads per warp, 16 lanes per head. A lane holds both members of its four rotary pairs, elements
    // [4 sub, +4) and [half + 4 sub, +4), or, past the rotated features, eight that pass through (two runs of
    // four at 2 half + 8 (sub - half / 4)); so the rotation needs no exchange between lanes, and the math runs
    // on packed fp32 pairs. Pass-through lanes rotate by cos 1, sin 0.
    const int sub = lane & 15, slot = lane >> 4, hp = half / 4;   // hp: lanes that hold rotary pairs
    const bool pairs = sub < hp;
    const int off0 = pairs ? 4 * sub : 2 * half + 8 * (sub - hp), off1 = pairs ? half + 4 * sub : off0 + 4;
    uint64_t wq2[4], wk2[4];   // norm weights of this lane's elements, packed in pairs
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = (i < 2 ? off0 : off1) + 2 * (i & 1);
      wq2[i] = norm ? f2_pack(a.q_norm_w[e], a.q_norm_w[e + 1]) : f2_pack(1.f, 1.f);
      wk2[i] = norm ? f2_pack(a.k_norm_w[e], a.k_norm_w[e + 1]) : f2_pack(1.f, 1.f);
    }
    const int steps = (heads + 1) / 2;
    // warps below steps % 8 take one more round per token than the others; the cos/sin fill goes to the others
    // first (fill index fi: threads rotated so that warp steps % 8 starts at 0), off the token's critical path
    const int fi = (warp * 32 + lane + 256 - 32 * (steps % 8)) & 255;
    for (int kk = 0; kk < n_mine; ++kk) {
      const int t = blockIdx.x + kk * gridDim.x;
      const int s = kk % KB_STAGES;
      uint8_t* st = kb_smem + s * L.bytes;
      if (FUSED && kk % KB_META == 0) {
        // the next KB_META tokens' row, position (and length) into shared memory, one token per thread: their
        // loads overlap, instead of one dependent global load at the head of every token (the table fill and
        // the barrier after it would wait for each). Entries are rewritten only here, after every computing
        // thread has passed the previous token's barrier, and each token's entries are read before it.
        const int i = warp * 32 + lane;
        if (i < KB_META && kk + i < n_mine) {
          const int ti = blockIdx.x + (kk + i) * gridDim.x;
          meta_row[i] = a.rows[ti];
          meta_pos[i] = a.positions[ti];
          meta_len[i] = f.use_seq_len ? a.seq_len[ti] : 0;
        }
        asm volatile("bar.sync 2, 256;" ::: "memory");
      }
      int row = 0, pos = 0, len = 0;
      const bool tabler = FUSED && fi < half;   // forms one of this token's cos/sin pairs
      if (FUSED) {
        const int mi = kk % KB_META;
        if (warp == 0 && lane == 0) row = meta_row[mi];
        if (tabler || (warp == 0 && lane == 0)) pos = meta_pos[mi];
        if (tabler) len = meta_len[mi];
      } else {
        if (warp == 0 && lane == 0) row = a.rows[t];
        if (warp == 0 && lane == 0) pos = a.positions[t];
      }
      if (FUSED) {
        // this token's cos/sin into the stage, one rotary pair per computing thread (the tables' arithmetic);
        // that part of the stage is not copied in, and the barrier below keeps the warps within one token, so
        // the previous use of this stage has been read
        const int i = fi;
        if (i < half) {
          const bool use_long = f.use_seq_len && len > f.switch_len;
          const unsigned long long turn = use_long ? f.turn_long[i] : f.turn_short[i];
          const unsigned long long frac = static_cast<unsigned long long>(pos) * turn;   // mod 2^64
          const int top = static_cast<int>(static_cast<unsigned int>(frac >> 32));
          float cv, sv;
          sincospif(static_cast<float>(top) * 4.656612873077393e-10f, &sv, &cv);
          reinterpret_cast<float*>(st + L.cos)[i] = pos < 0 ? 0.f : cv * f.af;
          reinterpret_cast<float*>(st + L.sin)[i] = pos < 0 ? 0.f : sv * f.af;
          if (pos < 0 && i == 0) set_error(a.err, kErrIndex);
        }
      }
      if (FUSED) {
        // every computing warp goes on, or all leave together (a warp alone at the barrier would wait forever);
        // the barrier also orders the cos/sin above before their reads
        uint32_t all_ok;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(all_ok)
            : "r"(mbar_wait(full(s), (kk / KB_STAGES) & 1, a.err) ? 1u : 0u)
            : "memory");
        if (!all_ok) break;
      } else if (!__all_sync(0xffffffffu, mbar_wait(full(s), (kk / KB_STAGES) & 1, a.err))) {
        break;
      }
      if (warp == 0 && lane == 0) {
        // the token's cache slot, for the copy thread (published by this thread's arrival on done[s]); written
        // only now: the stage's full barrier is armed after the copy thread has read the previous token's slot
        const long long slot_ = kv_slot(kv_layout(a), row, pos);
        if (slot_ < 0) set_error(a.err, kErrIndex);
        *reinterpret_cast<long long*>(st + L.hdr) = slot_;
      }
      uint64_t c2[2], s2[2];   // cos / sin of this lane's pairs 4 sub .. 4 sub + 3
      if (pairs) {
        const float4 c4 = *reinterpret_cast<const float4*>(st + L.cos + 4 * sub * 4);
        const float4 s4 = *reinterpret_cast<const float4*>(st + L.sin + 4 * sub * 4);
        c2[0] = f2_pack(c4.x, c4.y); c2[1] = f2_pack(c4.z, c4.w);
        s2[0] = f2_pack(-s4.x, -s4.y); s2[1] = f2_pack(-s4.z, -s4.w);   // negated: y_lo = x_lo c - x_hi s
      } else {
        c2[0] = c2[1] = f2_pack(1.f, 1.f);
        s2[0] = s2[1] = f2_pack(0.f, 0.f);
      }
      for (int step = warp; step < steps; step += 8) {
        const int hh = step * 2 + slot;
        const bool live = hh < heads;
        const bool is_q = hh < a.hq;
        uint8_t* vec = st + (is_q ? hh * D * 2 : L.k + (hh - a.hq) * D * 2);
        uint2 lo = make_uint2(0u, 0u), hi = make_uint2(0u, 0u);
        if (live) {
          lo = *reinterpret_cast<const uint2*>(vec + off0 * 2);
          hi = *reinterpret_cast<const uint2*>(vec + off1 * 2);
        }
        // bf16 -> fp32 pairs: a bf16 is the high half of its fp32
        uint64_t x2[4] = {f2_pack(__uint_as_float(lo.x << 16), __uint_as_float(lo.x & 0xffff0000u)),
                          f2_pack(__uint_as_float(lo.y << 16), __uint_as_float(lo.y & 0xffff0000u)),
                          f2_pack(__uint_as_float(hi.x << 16), __uint_as_float(hi.x & 0xffff0000u)),
                          f2_pack(__uint_as_float(hi.y << 16), __uint_as_float(hi.y & 0xffff0000u))};
        if (norm) {
          uint64_t q2 = f2_mul(x2[0], x2[0]);
#pragma unroll
          for (int i = 1; i < 4; ++i) q2 = f2_fma(x2[i], x2[i], q2);
          float q0, q1;
          f2_unpack(q2, q0, q1);
          float ss = q0 + q1;
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          const float rs = rsqrtf(ss * (1.0f / D) + a.eps);
          const uint64_t rs2 = f2_pack(rs, rs);
#pragma unroll
          for (int i = 0; i < 4; ++i) x2[i] = f2_mul(f2_mul(x2[i], rs2), is_q ? wq2[i] : wk2[i]);
        }
        // y_lo = x_lo c - x_hi s, y_hi = x_hi c + x_lo s
        uint64_t y2[4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          y2[i] = f2_fma(x2[2 + i], s2[i], f2_mul(x2[i], c2[i]));
          y2[2 + i] = f2_fma(x2[i], f2_mul(s2[i], f2_pack(-1.f, -1.f)), f2_mul(x2[2 + i], c2[i]));
        }
        if (live) {
          float f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) f2_unpack(y2[i], f[2 * i], f[2 * i + 1]);
          *reinterpret_cast<uint2*>(vec + off0 * 2) = make_uint2(bf16x2_bits(f[0], f[1]), bf16x2_bits(f[2], f[3]));
          *reinterpret_cast<uint2*>(vec + off1 * 2) = make_uint2(bf16x2_bits(f[4], f[5]), bf16x2_bits(f[6], f[7]));
        }
      }
      fence_proxy_async_smem();   // the rotated vectors (generic proxy) -> visible to the bulk stores
      mbar_arrive(done(s));
    }
    return;
  } else {
    const int sub = lane % TPV, slot = lane / TPV, e0 = sub * VEC;
    const int hc = half / VEC;
    const bool lower = sub < hc, upper = sub >= hc && sub < 2 * hc;
    const int psub = lower ? sub + hc : (upper ? sub - hc : sub);
    const int src_lane = slot * TPV + psub;
    const int ci = (lower ? sub : sub - hc) * VEC;   // this piece's pairs (lower or upper half)
    const bool norm = a.q_norm_w != nullptr;
    float wq[VEC], wk[VEC];
    if (norm) {
  #pragma unroll
      for (int j = 0; j < VEC; j += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(a.q_norm_w + e0 + j);
        const float4 k4 = *reinterpret_cast<const float4*>(a.k_norm_w + e0 + j);
        wq[j] = q4.x; wq[j + 1] = q4.y; wq[j + 2] = q4.z; wq[j + 3] = q4.w;
        wk[j] = k4.x; wk[j + 1] = k4.y; wk[j + 2] = k4.z; wk[j + 3] = k4.w;
      }
    }
    const int steps = (heads + HPW - 1) / HPW;
    for (int kk = 0; kk < n_mine; ++kk) {
      const int t = blockIdx.x + kk * gridDim.x;
      const int s = kk % KB_STAGES;
      uint8_t* st = kb_smem + s * L.bytes;
      int row = 0, pos = 0;
      if (warp == 0 && lane == 0) {
        row = a.rows[t];
        pos = a.positions[t];
      }
      if (!__all_sync(0xffffffffu, mbar_wait(full(s), (kk / KB_STAGES) & 1, a.err))) break;
      if (warp == 0 && lane == 0) {
        // the token's cache slot, for the copy thread (published by this thread's arrival on done[s]); written
        // only now: the stage's full barrier is armed after the copy thread has read the previous token's slot
        const long long slot = kv_slot(kv_layout(a), row, pos);
        if (slot < 0) set_error(a.err, kErrIndex);
        *reinterpret_cast<long long*>(st + L.hdr) = slot;
      }
      float c[VEC], sv[VEC];
      if (lower || upper) {
  #pragma unroll
        for (int j = 0; j < VEC; j += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(st + L.cos + (ci + j) * 4);
          const float4 s4 = *reinterpret_cast<const float4*>(st + L.sin + (ci + j) * 4);
          c[j] = c4.x; c[j + 1] = c4.y; c[j + 2] = c4.z; c[j + 3] = c4.w;
          sv[j] = s4.x; sv[j + 1] = s4.y; sv[j + 2] = s4.z; sv[j + 3] = s4.w;
        }
      }
      for (int step = warp; step < steps; step += 8) {
        const int hh = step * HPW + slot;
        const bool live = hh < heads;
        const bool is_q = hh < a.hq;
        T* vec = reinterpret_cast<T*>(st + (is_q ? hh * D * es : L.k + (hh - a.hq) * D * es)) + e0;
        float x[VEC];
        if (live) V::load(vec, x);
        else {
  #pragma unroll
          for (int j = 0; j < VEC; ++j) x[j] = 0.f;
        }
        if (norm) {
          float ss = 0.f;
  #pragma unroll
          for (int j = 0; j < VEC; ++j) ss = fmaf(x[j], x[j], ss);
  #pragma unroll
          for (int off = TPV / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off, TPV);
          const float rs = rsqrtf(ss * (1.0f / D) + a.eps);
  #pragma unroll
          for (int j = 0; j < VEC; ++j) x[j] = x[j] * rs * (is_q ? wq[j] : wk[j]);
        }
        float px[VEC], y[VEC];
  #pragma unroll
        for (int j = 0; j < VEC; ++j) px[j] = __shfl_sync(0xffffffffu, x[j], src_lane);
        if (lower || upper) {
          const float sgn = lower ? -1.f : 1.f;
  #pragma unroll
          for (int j = 0; j < VEC; ++j) y[j] = fmaf(sgn * px[j], sv[j], x[j] * c[j]);
        } else {
  #pragma unroll
          for (int j = 0; j < VEC; ++j) y[j] = x[j];
        }
        if (live) V::store(vec, y);
      }
      fence_proxy_async_smem();   // the rotated vectors (generic proxy) -> visible to the bulk stores
      mbar_arrive(done(s));
    }
  }
}

template <typename T, int D, bool FUSED>
static cudaError_t launch_bulk(const KvUpdateArgs& a, const KbLayout& L, const RopeTurns& f, int smem,
                               cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kv_update_bulk_kernel<T, D, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int per_sm = 0, dev = 0, n_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kv_update_bulk_kernel<T, D, FUSED>, KB_THREADS, smem);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(a.n, n_sm * std::max(per_sm, 1)));
  return launch_dependent(kv_update_bulk_kernel<T, D, FUSED>, dim3(grid), dim3(KB_THREADS), smem, stream, a, L, f);
}

template <typename T, int D>
static cudaError_t launch_kv_t(const KvUpdateArgs& a, cudaStream_t stream) {
  if (a.n == 0) return cudaSuccess;
  // warps per token: enough warps in the grid (~2048) to cover memory latency, at most one per head group
  constexpr int HPW = 32 / (D / Vec16<T>::N);
  const int groups = (a.hq + a.hkv + HPW - 1) / HPW;
  KvUpdateArgs b = a;
  b.wpt = std::max(1, std::min(groups, (2048 + a.n - 1) / a.n));
  constexpr int VEC = Vec16<T>::N;
  const int half = a.rot / 2;
  if (half % VEC == 0 && half % 4 == 0) {
    const KbLayout L = kb_layout(a.hq, a.hkv, D, half, static_cast<int>(sizeof(T)));
    const int smem = KB_STAGES * L.bytes;
    if (smem <= 200 * 1024) {
      return launch_bulk<T, D, false>(a, L, RopeTurns{}, smem, stream);
    }
  }
  const long long warps = static_cast<long long>(a.n) * b.wpt;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);   // 8 warps per block
  if ((a.rot / 2) % Vec16<T>::N == 0)
    return launch_dependent(kv_update_kernel<T, D, true>, dim3(blocks), dim3(256), 0, stream, b);
  return launch_dependent(kv_update_kernel<T, D, false>, dim3(blocks), dim3(256), 0, stream, b);
}

cudaError_t launch_kv_update(const KvUpdateArgs& a, bool bf16, cudaStream_t stream) {
  if (bf16) return a.d == 64 ? launch_kv_t<__nv_bfloat16, 64>(a, stream) : launch_kv_t<__nv_bfloat16, 128>(a, stream);
  return a.d == 64 ? launch_kv_t<float, 64>(a, stream) : launch_kv_t<float, 128>(a, stream);
}

bool kv_update_rope_supported(bool bf16, int d, int rot) {
  return bf16 && d == 128 && (rot / 2) % 8 == 0;
}

cudaError_t launch_kv_update_rope(const KvUpdateArgs& a, const RopeFreqs& freqs, cudaStream_t stream) {
  if (a.n == 0) return cudaSuccess;
  const int half = a.rot / 2;
  const KbLayout L = kb_layout(a.hq, a.hkv, 128, half, 2);
  const int smem = KB_STAGES * L.bytes;
  if (!kv_update_rope_supported(true, a.d, a.rot) || smem > 200 * 1024) return cudaErrorNotSupported;
  return launch_bulk<__nv_bfloat16, 128, true>(a, L, rope_turns(freqs), smem, stream);
}

}  // namespace da
