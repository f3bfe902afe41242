// Split-K decode attention for bf16 caches, head_dim 128, GQA groups of up to 8 query heads.
//
// One new token per sequence attends over its cache row: the decode case of DecoderAttention.forward
// (page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", sections
// "What differs between model families" and "Sliding windows": on a windowed layer only the last w
// keys are read, so the cost per token is O(w) however long the context).
//
// The step is bound by HBM: every visible key costs 2 * Hkv * d * 2 bytes (K and V) and is read once.
// Work unit = (key chunk, KV head, sequence): one CTA streams its chunk of K and V through a ring of
// TMA-filled shared-memory stages (128-byte swizzled tiles of 64 keys) and serves all G = Hq/Hkv query
// heads of the group from each tile, so K/V bytes are read once per group, not once per head.
// Scores S^T = K Q^T and the update O^T += V^T P^T run as m16n8k16 bf16 MMAs with the keys (then the head
// dims) on the M side and the (padded) query group on N; the softmax is fp32 with warp-shuffle max/sum.
// Each CTA writes its partial (max, sum, unnormalised output) per head to the workspace; a merge kernel
// combines the chunks of a (sequence, head) in a fixed order.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {
namespace dec {

constexpr int BK = 64;                  // keys per tile
constexpr int D = 128;
constexpr int CWARPS = 4;               // compute warps; each takes 16 keys of a tile
constexpr int THREADS = (CWARPS + 1) * 32;
constexpr int HALF_BYTES = BK * 128;    // one 64-wide half of a tile: 64 rows x 128 B = 8 KB
constexpr int TILE_BYTES = 2 * HALF_BYTES;
constexpr int STAGE_BYTES = 2 * TILE_BYTES;   // K tile + V tile = 32 KB
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const __nv_bfloat16* q_rot;
  const int32_t* rows;
  const int32_t* positions;
  float* ws_o;        // [S, Hq, n_splits, D]
  float2* ws_ml;      // [S, Hq, n_splits] (max in log2 units, sum)
  __nv_bfloat16* out; // [S, Hq, D]
  int hq, hkv, max_len, num_rows, window;
  float softcap, scale;
  const float* sinks;   // [Hq] sink logits (natural units) or NULL
  const int32_t* block_table;   // paged pool: [num_rows, max_blocks] block ids; NULL: contiguous cache
  int block_size, max_blocks, n_blocks;
  int chunk, n_splits;
  int* err;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset, inside a K or V tile, of the 16-byte chunk `c16` (0..15 along d) of key row `r`
// (0..63) under the 128-byte swizzle TMA applies to each 64-wide half.
__device__ __forceinline__ uint32_t sw_off(int r, int c16) {
  return static_cast<uint32_t>((c16 >> 3) * HALF_BYTES + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

// Keys [lo, p] of the sequence are visible. Chunk c covers [base + c*chunk, min(base + (c+1)*chunk, p+1)):
// base = lo for a contiguous cache; for a paged pool lo rounded down to a multiple of the 64-key tile, so
// that a tile never straddles two blocks (block sizes are multiples of 64), the keys below lo masked.
__device__ __forceinline__ void key_range(int p, int window, bool paged, int& lo, int& base, int& n_span) {
  lo = window > 0 ? max(0, p + 1 - window) : 0;
  base = paged ? (lo & ~(BK - 1)) : lo;
  n_span = p + 1 - base;
}

template <int NST>
__global__ void __launch_bounds__(THREADS) decode_kernel(const __grid_constant__ CUtensorMap tmk,
                                                         const __grid_constant__ CUtensorMap tmv, const Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * STAGE_BYTES);   // full[NST], empty[NST]
  __shared__ float comb_m[CWARPS][8], comb_l[CWARPS][8];

  const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();   // the stream's previous kernel (the cache update) has finished writing the caches
  const int p = prm.positions[s];
  const int row = prm.rows[s];
  if (row < 0 || row >= prm.num_rows || p < 0 || p >= prm.max_len) {
    if (threadIdx.x == 0 && c == 0 && g == 0) set_error(prm.err, kErrIndex);
    return;   // the merge kernel writes zeros for this sequence
  }
  int lo, base, n_span;
  key_range(p, prm.window, prm.block_table != nullptr, lo, base, n_span);
  const int k0 = base + c * prm.chunk;
  if (k0 > p) return;                       // this sequence has fewer chunks
  const int k1 = min(k0 + prm.chunk, p + 1);
  const int n_tiles = (k1 - k0 + BK - 1) / BK;
  const int G = prm.hq / prm.hkv;
  const int h0 = g * G;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int st) { return bar0 + 8u * st; };
  auto empty_bar = [&](int st) { return bar0 + 8u * (NST + st); };
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), CWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == CWARPS) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      const uint64_t pol = policy_evict_first();
      const KvLayout kvl = kv_layout(prm);
      const long long plane = (static_cast<long long>(row) * prm.hkv + g) * prm.max_len;   // contiguous
      const long long head_off = g * kv_head_stride(kvl);                                    // paged
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(empty_bar(st), ((i / NST) + 1) & 1, prm.err)) break;
        const uint32_t dst = sbase + st * STAGE_BYTES;
        mbar_arrive_expect_tx(full_bar(st), STAGE_BYTES);
        long long slot = plane + k0 + i * BK;
        if (prm.block_table) {   // the tile's 64 keys lie in one block
          slot = kv_slot(kvl, row, k0 + i * BK);
          if (slot < 0) {        // no block: reported; a slot inside the pool keeps the copy's byte count
            set_error(prm.err, kErrIndex);
            slot = 0;
          }
          slot += head_off;
        }
        const int key = static_cast<int>(slot);
        tma_load_2d_hint(dst, &tmk, full_bar(st), 0, key, pol);
        tma_load_2d_hint(dst + HALF_BYTES, &tmk, full_bar(st), 64, key, pol);
        tma_load_2d_hint(dst + TILE_BYTES, &tmv, full_bar(st), 0, key, pol);
        tma_load_2d_hint(dst + TILE_BYTES + HALF_BYTES, &tmv, full_bar(st), 64, key, pol);
        ++issued;
      }
      // drain: the last load of each stage must have landed before the CTA may exit
      for (int i = max(0, issued - NST); i < issued; ++i) mbar_wait(full_bar(i % NST), (i / NST) & 1, prm.err);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers (4 warps)
  const int gq = lane >> 2, cq = lane & 3;
  // B operand (Q^T, k = d, n = head): b0 = Q[h0+gq][16kk + 2cq .. +1], b1 = same at +8
  uint32_t qb[8][2];
  {
    const bool hv = gq < G;
    const __nv_bfloat16* qrow = prm.q_rot + (static_cast<long long>(s) * prm.hq + h0 + (hv ? gq : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qb[kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * cq) : 0u;
      qb[kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * cq) : 0u;
    }
  }
  const float cap = prm.softcap;
  const float zmul = cap > 0.f ? prm.scale / cap : prm.scale * kLog2e;
  const float cap_l2 = cap * kLog2e;

  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % NST;
    if (!mbar_wait(full_bar(st), (i / NST) & 1, prm.err)) { ok = false; break; }
    const uint32_t sK = sbase + st * STAGE_BYTES;
    const uint32_t sV = sK + TILE_BYTES;
    const int kb = k0 + i * BK + warp * 16;        // first key of this warp's 16
    const int n_valid = k1 - kb;                   // keys of the 16 that are in the chunk (may be <= 0)
    const int n_lo = lo - kb;                      // keys of the 16 below the window (paged tiles only)

    // S^T[16 keys x 8 heads]
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3, r8 = lane & 7;
      const int kr = warp * 16 + (mi & 1) * 8 + r8;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sK + sw_off(kr, kk * 2 + (mi >> 1)), a0, a1, a2, a3);
        mma_16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
    }
    // logits in log2 units, masked
    const bool v0 = gq >= n_lo && gq < n_valid, v1 = gq + 8 >= n_lo && gq + 8 < n_valid;
    float z[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float t = sc[e] * zmul;
      if (cap > 0.f) t = cap_l2 * tanh_fast(t);
      z[e] = ((e < 2) ? v0 : v1) ? t : -CUDART_INF_F;
    }
    float tmax[2] = {fmaxf(z[0], z[2]), fmaxf(z[1], z[3])};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 4));
      tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 8));
      tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 16));
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float mn = fmaxf(m_run[j], tmax[j]);
      muse[j] = (mn == -CUDART_INF_F) ? 0.f : mn;
      alpha[j] = ex2(m_run[j] - muse[j]);
      m_run[j] = mn;
    }
    const float p0 = ex2(z[0] - muse[0]), p1 = ex2(z[1] - muse[1]);
    const float p2 = ex2(z[2] - muse[0]), p3 = ex2(z[3] - muse[1]);
    l_run[0] = l_run[0] * alpha[0] + p0 + p2;
    l_run[1] = l_run[1] * alpha[1] + p1 + p3;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= alpha[0];
      o[mt][1] *= alpha[1];
      o[mt][2] *= alpha[0];
      o[mt][3] *= alpha[1];
    }
    // P^T as the B operand (k = key, n = head): transpose the 8x8 blocks of P^T held row-major
    const uint32_t b0 = movmatrix_t(pack_bf16(p0, p1));
    const uint32_t b1 = movmatrix_t(pack_bf16(p2, p3));
    // O^T[d x heads] += V^T[d x 16 keys] P^T[16 keys x heads]
    {
      const int mi = lane >> 3, r8 = lane & 7;
      const int vr = warp * 16 + (mi >> 1) * 8 + r8;
      const bool partial = n_valid < 16 || n_lo > 0;
      // keys this thread's A-fragment halves belong to: 2cq, 2cq+1 (regs 0,1) and 8+2cq, 9+2cq (regs 2,3)
      auto in = [&](int k) { return k >= n_lo && k < n_valid; };
      const uint32_t keep01 = (in(2 * cq) ? 0x0000ffffu : 0u) | (in(2 * cq + 1) ? 0xffff0000u : 0u);
      const uint32_t keep23 = (in(2 * cq + 8) ? 0x0000ffffu : 0u) | (in(2 * cq + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(sV + sw_off(vr, mt * 2 + (mi & 1)), a0, a1, a2, a3);
        if (partial) {   // slots past the chunk may hold anything (even NaN): 0 * NaN must not reach O
          a0 &= keep01;
          a1 &= keep01;
          a2 &= keep23;
          a3 &= keep23;
        }
        mma_16816(o[mt], a0, a1, a2, a3, b0, b1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(st));
  }

  // -------------------------------------------------------------------- combine the 4 warps
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
  }
  if (gq == 0) {
    comb_m[warp][2 * cq] = m_run[0];
    comb_m[warp][2 * cq + 1] = m_run[1];
    comb_l[warp][2 * cq] = l_run[0];
    comb_l[warp][2 * cq + 1] = l_run[1];
  }
  // all stages are consumed: reuse stage memory for the per-warp outputs [warp][head][d]
  asm volatile("bar.sync 1, %0;" ::"n"(CWARPS * 32) : "memory");
  float* comb_o = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int dd = mt * 16 + gq;
    comb_o[(warp * 8 + 2 * cq) * D + dd] = o[mt][0];
    comb_o[(warp * 8 + 2 * cq + 1) * D + dd] = o[mt][1];
    comb_o[(warp * 8 + 2 * cq) * D + dd + 8] = o[mt][2];
    comb_o[(warp * 8 + 2 * cq + 1) * D + dd + 8] = o[mt][3];
  }
  asm volatile("bar.sync 1, %0;" ::"n"(CWARPS * 32) : "memory");
  if (!ok) return;
  const int dd = threadIdx.x;   // 0..127
  for (int n = 0; n < G; ++n) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < CWARPS; ++w) M = fmaxf(M, comb_m[w][n]);
    const float Mu = (M == -CUDART_INF_F) ? 0.f : M;
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < CWARPS; ++w) {
      const float wt = ex2(comb_m[w][n] - Mu);
      acc += wt * comb_o[(w * 8 + n) * D + dd];
      L += wt * comb_l[w][n];
    }
    const long long slot = (static_cast<long long>(s) * prm.hq + h0 + n) * prm.n_splits + c;
    prm.ws_o[slot * D + dd] = acc;
    if (dd == 0) prm.ws_ml[slot] = make_float2(M, L);
  }
}

// One block of D threads per (query head, sequence): combine the chunks in order.
__global__ void __launch_bounds__(D) merge_kernel(const Params prm) {
  const int h = blockIdx.x, s = blockIdx.y, dd = threadIdx.x;
  __nv_bfloat16* out = prm.out + (static_cast<long long>(s) * prm.hq + h) * D;
  pdl_wait();   // the decode kernel's partial results are complete
  const int p = prm.positions[s];
  const int row = prm.rows[s];
  if (row < 0 || row >= prm.num_rows || p < 0 || p >= prm.max_len) {
    out[dd] = __float2bfloat16_rn(0.f);
    return;
  }
  int lo, k_base, n_span;
  key_range(p, prm.window, prm.block_table != nullptr, lo, k_base, n_span);
  const int n_spl = (n_span + prm.chunk - 1) / prm.chunk;
  const long long base = (static_cast<long long>(s) * prm.hq + h) * prm.n_splits;
  float M = -CUDART_INF_F;
  for (int c = 0; c < n_spl; ++c) M = fmaxf(M, prm.ws_ml[base + c].x);
  const float sink = prm.sinks ? prm.sinks[h] * kLog2e : -CUDART_INF_F;   // log2 units, like the partials
  M = fmaxf(M, sink);
  const float Mu = (M == -CUDART_INF_F) ? 0.f : M;
  float acc = 0.f, L = prm.sinks ? ex2(sink - Mu) : 0.f;   // the sink's share joins the sum, no value
  for (int c = 0; c < n_spl; ++c) {
    const float2 ml = prm.ws_ml[base + c];
    const float wt = ex2(ml.x - Mu);
    acc += wt * prm.ws_o[(base + c) * D + dd];
    L += wt * ml.y;
  }
  out[dd] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
}

}  // namespace dec

// Scratch of da_attn_decode_noalloc: a fixed array in the module's global memory, so that callers who
// may not allocate device memory can still run the split-K decode. Every GPU that loads the library holds
// these bytes until the process exits. Host code must not pass the symbol itself to a kernel (on the host
// it names a stand-in, not device memory): static_scratch() looks up its device address once per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeStaticScratchBytes];

void* static_scratch() {
  static std::mutex mu;
  static void* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

DecodePlan decode_plan(int hkv, int n_seqs, int max_len, int window, bool aligned) {
  DecodePlan p;
  // keys a chunk sequence spans at most (aligned: from the window start rounded down to a 64-key tile)
  const int max_keys = (window > 0 ? std::min(window, max_len) : max_len) + (aligned ? dec::BK - 1 : 0);
  int chunk = 512;
#ifdef DA_TUNING_HOOKS
  const char* env = std::getenv("DA_DECODE_CHUNK");   // sweep override in tuning builds only (multiple of 64)
  if (env && std::atoi(env) >= 64 && std::atoi(env) % 64 == 0) {
    chunk = std::atoi(env);
  } else
#endif
  {
    // Grow the chunk (fewer partials to write and merge) while the grid keeps >= 8 CTAs per SM of a
    // 152-SM GB300 busy.
    const long long target = 152LL * 8;
    while (chunk < 4096 && static_cast<long long>(n_seqs) * hkv * ((max_keys + 2 * chunk - 1) / (2 * chunk)) >= target)
      chunk *= 2;
  }
  p.chunk = chunk;
  p.n_splits = std::max(1, (max_keys + chunk - 1) / chunk);
  return p;
}

size_t decode_workspace_bytes(int hq, int n_seqs, const DecodePlan& p) {
  const size_t per = static_cast<size_t>(dec::D) * sizeof(float) + sizeof(float2);
  return static_cast<size_t>(n_seqs) * hq * p.n_splits * per + 256;
}

cudaError_t launch_decode_bf16(const AttnArgs& a, const DecodePlan& plan, void* workspace, cudaStream_t stream) {
  using namespace dec;
  if (a.n_seqs == 0) return cudaSuccess;
  constexpr int NST = 3;
  CUtensorMap tmk, tmv;
  const uint64_t rows_total = a.block_table ? static_cast<uint64_t>(a.n_blocks) * a.hkv * a.block_size
                                            : static_cast<uint64_t>(a.num_rows) * a.hkv * a.max_len;
  if (!encode_tmap_2d_bf16(&tmk, a.k_cache, D, rows_total, D * 2, 64, BK) ||
      !encode_tmap_2d_bf16(&tmv, a.v_cache, D, rows_total, D * 2, 64, BK))
    return cudaErrorInvalidValue;
  Params prm;
  prm.q_rot = static_cast<const __nv_bfloat16*>(a.q_rot);
  prm.rows = a.rows;
  prm.positions = a.positions;
  const size_t o_bytes = static_cast<size_t>(a.n_seqs) * a.hq * plan.n_splits * D * sizeof(float);
  prm.ws_o = static_cast<float*>(workspace);
  prm.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + ((o_bytes + 255) & ~size_t(255)));
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.hq = a.hq;
  prm.hkv = a.hkv;
  prm.max_len = a.max_len;
  prm.num_rows = a.num_rows;
  prm.window = a.window;
  prm.softcap = a.softcap;
  prm.sinks = a.sinks;
  prm.block_table = a.block_table;
  prm.block_size = a.block_size;
  prm.max_blocks = a.max_blocks;
  prm.n_blocks = a.n_blocks;
  prm.scale = a.scale;
  prm.chunk = plan.chunk;
  prm.n_splits = plan.n_splits;
  prm.err = a.err;
  const int smem = NST * STAGE_BYTES + 2 * NST * 8 + 1024;
  // per device and cheap: set on every launch, so that a call on any device (or host thread) finds it
  cudaError_t ea = cudaFuncSetAttribute(decode_kernel<NST>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (ea != cudaSuccess) return ea;
  dim3 grid(plan.n_splits, a.hkv, a.n_seqs);
  cudaError_t e = launch_dependent(decode_kernel<NST>, grid, dim3(THREADS), smem, stream, tmk, tmv, prm);
  if (e != cudaSuccess) return e;
  return launch_dependent(merge_kernel, dim3(a.hq, a.n_seqs), dim3(D), 0, stream, prm);
}

}  // namespace da
