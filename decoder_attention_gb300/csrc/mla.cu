// Multi-head latent attention (MLA) decode with absorbed up-projections, bf16, latent rank 512, rotary 64.
//
// Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", section "Multi-head
// latent attention" and "Serving it: absorbing the up-projections": each token caches one row [c, k_rope]
// of 576 numbers; every query head arrives already mapped into latent space (q = [W_uk^T q_nope, q_rope]),
// so decode is multi-query attention of all heads against the cached rows, whose first 512 features are
// the values. The output is the latent (512 wide) per head; W_uv is applied outside.
//
// mla_update_kernel writes the rows (rotary part deinterleaved from DeepSeek's adjacent pairs and rotated by
// the split-half rotation) and rotates the rotary part of the queries in place.
//
// mla_decode_kernel: work unit = (key chunk, group of 32 query heads, sequence). One producer warp streams the
// chunk's rows through a 3-stage ring of TMA-filled tiles (64 keys x 576, nine 128-byte-swizzled boxes of 64
// features); four compute warps share each 16-key slab with m16n8k16 bf16 MMAs: warp w computes partial scores
// S^T = K Q^T over features [144w, 144w + 144) for all 32 heads (its queries in registers), warp w sums the
// partials of heads 8w .. 8w + 7 and runs their online softmax, and warp w updates O^T for value features
// [128w, 128w + 128) of all 32 heads (O^T in registers), so every tile byte is read from shared memory once.
// The running max moves only when it grows by more than 2^8, so O is rescaled on few slabs. Each warp writes
// its partials (max, sum, unnormalised output); mla_merge_kernel combines the chunks in a fixed order.
//
// Roofline: a key costs 1152 bytes and H * (576 + 512) * 2 FLOP (278.5 KFLOP at H = 128, 242 FLOP per byte).
// At that intensity the step needs tensor-core rates well above what the legacy MMAs give (about 1600 FLOP
// per clock per SM, a fifth of tcgen05): this kernel is bound by MMA issue and latency, not by HBM.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {
namespace mla {

constexpr int RANK = 512;                 // latent width = value width
constexpr int ROPE = 64;                  // rotary width
constexpr int DR = RANK + ROPE;           // 576: a cached row
constexpr int BOXES = DR / 64;            // 9 boxes of 64 features per tile
constexpr int BK = 64;                    // keys per tile
constexpr int BOX_BYTES = BK * 128;       // 64 keys x 128 B = 8 KB
constexpr int STAGE_BYTES = BOXES * BOX_BYTES;   // 72 KB
constexpr int NST = 3;
constexpr int CWARPS = 4;                 // compute warps, 8 heads each
constexpr int HPW = 8;                    // heads per warp
constexpr int HPC = CWARPS * HPW;         // heads per CTA
constexpr int THREADS = (CWARPS + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
#ifndef DA_MLA_SACC
#define DA_MLA_SACC 4
#endif
constexpr int SACC = DA_MLA_SACC;   // independent partial sums of the 36-MMA score chain
constexpr float kGrow = 8.0f;       // log2 units: the running max may lag the true max by up to x256

struct Params {
  const __nv_bfloat16* q;     // [S, H, 576]
  const int32_t* rows;
  const int32_t* positions;
  float* ws_o;                // [S, H, n_splits, 512]
  float2* ws_ml;              // [S, H, n_splits] (max in log2 units, sum)
  __nv_bfloat16* out;         // [S, H, 512]
  int hq, max_len, num_rows, window;
  float scale;
  int chunk, n_splits;
  const int32_t* block_table;  // paged pool or NULL
  int block_size, max_blocks, n_blocks;
  int hkv;                     // 1 (one latent row per position), for the slot lookup
  int* err;
};

// Byte offset, inside a tile, of the 16-byte chunk c16 (0..71 along the 576 features) of key row r (0..63)
// under the 128-byte swizzle TMA applies to each 64-feature box.
__device__ __forceinline__ uint32_t sw_off(int r, int c16) {
  return static_cast<uint32_t>((c16 >> 3) * BOX_BYTES + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Keys [lo, p] are visible; chunks start at base (lo, rounded down to a 64-key tile for paged pools).
__device__ __forceinline__ void key_range(int p, int window, bool paged, int& lo, int& base, int& n_span) {
  lo = window > 0 ? max(0, p + 1 - window) : 0;
  base = paged ? (lo & ~(BK - 1)) : lo;
  n_span = p + 1 - base;
}

// ---------------------------------------------------------------------------------------------- update

struct UpdateParams {
  const __nv_bfloat16* latent;   // [N, 512]
  const __nv_bfloat16* k_rope;   // [N, 64], adjacent pairs
  const int32_t* rows;
  const int32_t* positions;
  const float* cos;              // [N, 32]
  const float* sin;
  __nv_bfloat16* q;              // [N, H, 576] or NULL: rotary part rotated in place
  __nv_bfloat16* cache;          // [rows_total, 576]
  int n, hq, num_rows, max_len;
  const int32_t* block_table;
  int block_size, max_blocks, n_blocks, hkv;
  int* err;
};

// One warp per (token, item): item 0 writes the token's cache row, item 1 + h rotates query head h.
// Pair i of the rotary features is (x[2i], x[2i+1]) in the checkpoint's order; deinterleaved it becomes
// (y[i], y[i + 32]), rotated: y'[i] = y[i] c_i - y[i+32] s_i, y'[i+32] = y[i+32] c_i + y[i] s_i.
__global__ void __launch_bounds__(256) mla_update_kernel(const UpdateParams a) {
  const int items = 1 + (a.q ? a.hq : 0);
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long long>(a.n) * items) return;
  pdl_wait();   // inputs written by the stream's previous kernel are visible
  const int t = static_cast<int>(w / items), item = static_cast<int>(w - static_cast<long long>(t) * items);
  const float c = a.cos[static_cast<long long>(t) * (ROPE / 2) + lane];
  const float s = a.sin[static_cast<long long>(t) * (ROPE / 2) + lane];
  if (item == 0) {
    const long long slot = kv_slot(kv_layout(a), a.rows[t], a.positions[t]);
    if (slot < 0) {
      if (lane == 0) set_error(a.err, kErrIndex);
      return;
    }
    __nv_bfloat16* dst = a.cache + slot * DR;
    const uint4* src = reinterpret_cast<const uint4*>(a.latent + static_cast<long long>(t) * RANK);
    reinterpret_cast<uint4*>(dst)[lane] = src[lane];             // 512 bf16 = 64 x 16 bytes
    reinterpret_cast<uint4*>(dst)[lane + 32] = src[lane + 32];
    const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162*>(a.k_rope + static_cast<long long>(t) * ROPE)[lane];
    const float x0 = __low2float(x), x1 = __high2float(x);
    dst[RANK + lane] = __float2bfloat16_rn(x0 * c - x1 * s);
    dst[RANK + 32 + lane] = __float2bfloat16_rn(x1 * c + x0 * s);
  } else {
    __nv_bfloat16* qr = a.q + (static_cast<long long>(t) * a.hq + (item - 1)) * DR + RANK;
    const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162*>(qr)[lane];
    const float x0 = __low2float(x), x1 = __high2float(x);
    __syncwarp();   // every lane has read its pair before any lane writes
    qr[lane] = __float2bfloat16_rn(x0 * c - x1 * s);
    qr[32 + lane] = __float2bfloat16_rn(x1 * c + x0 * s);
  }
}

// ---------------------------------------------------------------------------------------------- decode

__global__ void __launch_bounds__(THREADS, 1) mla_decode_kernel(const __grid_constant__ CUtensorMap tmc,
                                                                 const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * STAGE_BYTES);   // full[NST], empty[NST]
  volatile int* give_up = reinterpret_cast<volatile int*>(smem + NST * STAGE_BYTES + 64);

  const int c = blockIdx.x, hg = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();   // the stream's previous kernel (the cache update) has finished writing the cache
  const int p = prm.positions[s];
  const int row = prm.rows[s];
  if (row < 0 || row >= prm.num_rows || p < 0 || p >= prm.max_len) {
    if (threadIdx.x == 0 && c == 0 && hg == 0) set_error(prm.err, kErrIndex);
    return;   // the merge kernel writes zeros for this sequence
  }
  int lo, base, n_span;
  key_range(p, prm.window, prm.block_table != nullptr, lo, base, n_span);
  const int k0 = base + c * prm.chunk;
  if (k0 > p) return;
  const int k1 = min(k0 + prm.chunk, p + 1);
  const int n_tiles = (k1 - k0 + BK - 1) / BK;

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
      prefetch_tmap(&tmc);
      const KvLayout kvl = kv_layout(prm);
      const long long plane = static_cast<long long>(row) * prm.max_len;   // contiguous: rows [R * M, 576]
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(empty_bar(st), ((i / NST) + 1) & 1, prm.err)) break;
        const uint32_t dst = sbase + st * STAGE_BYTES;
        long long slot = plane + k0 + i * BK;
        if (prm.block_table) {   // the tile's 64 keys lie in one block
          slot = kv_slot(kvl, row, k0 + i * BK);
          if (slot < 0) {
            set_error(prm.err, kErrIndex);
            slot = 0;
          }
        }
        mbar_arrive_expect_tx(full_bar(st), STAGE_BYTES);
#pragma unroll
        for (int b = 0; b < BOXES; ++b)
          tma_load_2d(dst + b * BOX_BYTES, &tmc, full_bar(st), b * 64, static_cast<int>(slot));
        ++issued;
      }
      for (int i = max(0, issued - NST); i < issued; ++i) mbar_wait(full_bar(i % NST), (i / NST) & 1, prm.err);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  // Per 16-key slab: (1) warp w computes partial scores over features [144w, 144w + 144) for all 32 heads
  // (one A fragment feeds 4 MMAs) and stores them; (2) warp w sums the four partials of heads 8w .. 8w + 7,
  // runs their online softmax and stores P^T fragments and rescale factors; (3) warp w updates O^T for value
  // features [128w, 128w + 128) and all 32 heads (one A fragment feeds 4 MMAs). Every tile byte is read from
  // shared memory once per CTA.
  float* part = reinterpret_cast<float*>(smem + NST * STAGE_BYTES + 128);    // [4 warps][4 n-tiles][32][4]
  uint32_t* pfrag = reinterpret_cast<uint32_t*>(part + CWARPS * 4 * 32 * 4);  // [4 n-tiles][32][2]
  float* alpha_s = reinterpret_cast<float*>(pfrag + 4 * 32 * 2);             // [32 heads]
  volatile int* grow_s = reinterpret_cast<volatile int*>(alpha_s + 32);       // [4]: a head's max grew
  const int hbase = hg * HPC;
  const int gq = lane >> 2, cq = lane & 3;
  auto sync_compute = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(CWARPS * 32) : "memory"); };
  // B operands of the partial scores: heads hbase + 8nt + gq, features 144 warp + 16kk + 2cq (+8)
  uint32_t qb[4][9][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int h = min(hbase + nt * 8 + gq, prm.hq - 1);
    const __nv_bfloat16* qrow = prm.q + (static_cast<long long>(s) * prm.hq + h) * DR + warp * 144;
#pragma unroll
    for (int kk = 0; kk < 9; ++kk) {
      qb[nt][kk][0] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * cq);
      qb[nt][kk][1] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * cq);
    }
  }
  const float zmul = prm.scale * kLog2e;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};   // heads hbase + 8 warp + 2cq (+1)
  float l_run[2] = {0.f, 0.f};
  float o[8][4][4];                                   // O^T: features 128 warp + 16mt (+gq, +8), heads 8nt + 2cq (+1)
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;

  bool ok = true;
  const int mi = lane >> 3, r8 = lane & 7;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % NST;
    if (!__all_sync(0xffffffffu, mbar_wait(full_bar(st), (i / NST) & 1, prm.err))) ok = false;
    // the four warps agree on giving up, so that none waits at a barrier the others skip
    if (threadIdx.x == 0) *give_up = 0;
    sync_compute();
    if (!ok && lane == 0) *give_up = 1;
    sync_compute();
    if (*give_up) { ok = false; break; }
    const uint32_t sT = sbase + st * STAGE_BYTES;
    for (int slab = 0; slab < BK / 16; ++slab) {
      const int kb = k0 + i * BK + slab * 16;
      const int n_valid = k1 - kb;                   // uniform over the CTA
      if (n_valid <= 0) break;
      const int n_lo = lo - kb;
      // (1) partial scores
      float sp[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) sp[nt][0] = sp[nt][1] = sp[nt][2] = sp[nt][3] = 0.f;
      const int kr = slab * 16 + (mi & 1) * 8 + r8;
#pragma unroll
      for (int kk = 0; kk < 9; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sT + sw_off(kr, warp * 18 + kk * 2 + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_16816(sp[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        reinterpret_cast<float4*>(part)[(warp * 4 + nt) * 32 + lane] = make_float4(sp[nt][0], sp[nt][1], sp[nt][2], sp[nt][3]);
      sync_compute();
      // (2) softmax of heads 8 warp .. 8 warp + 7
      {
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < CWARPS; ++w) {
          const float4 v = reinterpret_cast<const float4*>(part)[(w * 4 + warp) * 32 + lane];
          sc[0] += v.x;
          sc[1] += v.y;
          sc[2] += v.z;
          sc[3] += v.w;
        }
        const bool v0 = gq >= n_lo && gq < n_valid, v1 = gq + 8 >= n_lo && gq + 8 < n_valid;
        float z[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) z[e] = ((e < 2) ? v0 : v1) ? sc[e] * zmul : -CUDART_INF_F;
        float tmax[2] = {fmaxf(z[0], z[2]), fmaxf(z[1], z[3])};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 4));
          tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 8));
          tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(0xffffffffu, tmax[j], 16));
        }
        // the running max moves only when it grows by more than kGrow (log2 units): P then stays below
        // 2^kGrow and O is rescaled on few slabs
        float alpha[2] = {1.f, 1.f}, muse[2];
        bool grow = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (tmax[j] > m_run[j] + kGrow) {
            alpha[j] = ex2(m_run[j] - tmax[j]);   // 0 while m_run is -inf
            m_run[j] = tmax[j];
            grow = true;
          }
          muse[j] = (m_run[j] == -CUDART_INF_F) ? 0.f : m_run[j];
        }
        const float p0 = ex2(z[0] - muse[0]), p1 = ex2(z[1] - muse[1]);
        const float p2 = ex2(z[2] - muse[0]), p3 = ex2(z[3] - muse[1]);
        l_run[0] = l_run[0] * alpha[0] + p0 + p2;
        l_run[1] = l_run[1] * alpha[1] + p1 + p3;
        reinterpret_cast<uint2*>(pfrag)[warp * 32 + lane] = make_uint2(movmatrix_t(pack2(p0, p1)), movmatrix_t(pack2(p2, p3)));
        if (gq == 0) {
          alpha_s[warp * 8 + 2 * cq] = alpha[0];
          alpha_s[warp * 8 + 2 * cq + 1] = alpha[1];
        }
        const bool any_grow = __any_sync(0xffffffffu, grow);   // written every slab, read after the barrier
        if (lane == 0) grow_s[warp] = any_grow ? 1 : 0;
      }
      sync_compute();
      // (3) O^T[128 features x 32 heads] += V^T P^T
      uint32_t pb[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint2 f = reinterpret_cast<const uint2*>(pfrag)[nt * 32 + lane];
        pb[nt][0] = f.x;
        pb[nt][1] = f.y;
      }
      if (grow_s[0] | grow_s[1] | grow_s[2] | grow_s[3]) {   // some head's max grew: rescale O (uniform)
        float al[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          al[nt][0] = alpha_s[nt * 8 + 2 * cq];
          al[nt][1] = alpha_s[nt * 8 + 2 * cq + 1];
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            o[mt][nt][0] *= al[nt][0];
            o[mt][nt][1] *= al[nt][1];
            o[mt][nt][2] *= al[nt][0];
            o[mt][nt][3] *= al[nt][1];
          }
      }
      const int vr = slab * 16 + (mi >> 1) * 8 + r8;
      const bool partial = n_valid < 16 || n_lo > 0;
      auto in = [&](int k) { return k >= n_lo && k < n_valid; };
      const uint32_t keep01 = (in(2 * cq) ? 0x0000ffffu : 0u) | (in(2 * cq + 1) ? 0xffff0000u : 0u);
      const uint32_t keep23 = (in(2 * cq + 8) ? 0x0000ffffu : 0u) | (in(2 * cq + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(sT + sw_off(vr, warp * 16 + mt * 2 + (mi & 1)), a0, a1, a2, a3);
        if (partial) {   // slots outside the chunk may hold anything (even NaN): 0 * NaN must not reach O
          a0 &= keep01;
          a1 &= keep01;
          a2 &= keep23;
          a3 &= keep23;
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mma_16816(o[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(st));
  }
  if (!ok) return;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
  }
  // (max, sum) of heads 8 warp + 2cq (+1); O^T features 128 warp + 16mt + gq (+8) of heads 8nt + 2cq (+1)
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int h = hbase + warp * 8 + 2 * cq + j;
    if (gq == 0 && h < prm.hq)
      prm.ws_ml[(static_cast<long long>(s) * prm.hq + h) * prm.n_splits + c] = make_float2(m_run[j], l_run[j]);
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = hbase + nt * 8 + 2 * cq + j;
      if (h >= prm.hq) continue;
      float* wo = prm.ws_o + ((static_cast<long long>(s) * prm.hq + h) * prm.n_splits + c) * RANK + warp * 128;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        wo[mt * 16 + gq] = o[mt][nt][j];
        wo[mt * 16 + gq + 8] = o[mt][nt][2 + j];
      }
    }
}

// One block of 128 threads per (query head, sequence): combine the chunks in order, 4 features a thread.
__global__ void __launch_bounds__(128) mla_merge_kernel(const Params prm) {
  const int h = blockIdx.x, s = blockIdx.y;
  __nv_bfloat16* out = prm.out + (static_cast<long long>(s) * prm.hq + h) * RANK;
  pdl_wait();   // the decode kernel's partial results are complete
  const int p = prm.positions[s];
  const int row = prm.rows[s];
  if (row < 0 || row >= prm.num_rows || p < 0 || p >= prm.max_len) {
    for (int f = threadIdx.x; f < RANK; f += blockDim.x) out[f] = __float2bfloat16_rn(0.f);
    return;
  }
  int lo, k_base, n_span;
  key_range(p, prm.window, prm.block_table != nullptr, lo, k_base, n_span);
  const int n_spl = (n_span + prm.chunk - 1) / prm.chunk;
  const long long base = (static_cast<long long>(s) * prm.hq + h) * prm.n_splits;
  float M = -CUDART_INF_F;
  for (int c = 0; c < n_spl; ++c) M = fmaxf(M, prm.ws_ml[base + c].x);
  const float Mu = (M == -CUDART_INF_F) ? 0.f : M;
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, L = 0.f;
  for (int c = 0; c < n_spl; ++c) {
    const float2 ml = prm.ws_ml[base + c];
    const float wt = ex2(ml.x - Mu);
    const float4 v = reinterpret_cast<const float4*>(prm.ws_o + (base + c) * RANK)[threadIdx.x];
    acc[0] += wt * v.x;
    acc[1] += wt * v.y;
    acc[2] += wt * v.z;
    acc[3] += wt * v.w;
    L += wt * ml.y;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint2 packed;
  packed.x = pack2(acc[0] * inv, acc[1] * inv);
  packed.y = pack2(acc[2] * inv, acc[3] * inv);
  reinterpret_cast<uint2*>(out)[threadIdx.x] = packed;
}

}  // namespace mla

MlaPlan mla_plan(int hq, int n_seqs, int max_len, int window, bool aligned) {
  MlaPlan p;
  const int max_keys = (window > 0 ? std::min(window, max_len) : max_len) + (aligned ? mla::BK - 1 : 0);
  if (hq == 128) {   // CTA-pair tcgen05 kernel
    p.chunk = mla_pair_chunk(n_seqs, max_keys);
    p.n_splits = std::max(1, (max_keys + p.chunk - 1) / p.chunk);
    return p;
  }
  const long long groups = static_cast<long long>(n_seqs) * ((hq + mla::HPC - 1) / mla::HPC);
  int chunk = 256;
  // grow the chunk (fewer partials) while the grid keeps >= 2 CTAs per SM of a 152-SM part
  while (chunk < 8192 && groups * ((max_keys + 2 * chunk - 1) / (2 * chunk)) >= 152LL * 2) chunk *= 2;
  p.chunk = chunk;
  p.n_splits = std::max(1, (max_keys + chunk - 1) / chunk);
  return p;
}

size_t mla_workspace_bytes(int hq, int n_seqs, const MlaPlan& p) {
  const size_t per = static_cast<size_t>(mla::RANK) * sizeof(float) + sizeof(float2);
  return static_cast<size_t>(n_seqs) * hq * p.n_splits * per + 256;
}

cudaError_t launch_mla_update(const MlaUpdateArgs& a, cudaStream_t stream) {
  using namespace mla;
  if (a.n == 0) return cudaSuccess;
  UpdateParams u;
  u.latent = static_cast<const __nv_bfloat16*>(a.latent);
  u.k_rope = static_cast<const __nv_bfloat16*>(a.k_rope);
  u.rows = a.rows;
  u.positions = a.positions;
  u.cos = a.cos;
  u.sin = a.sin;
  u.q = static_cast<__nv_bfloat16*>(a.q);
  u.cache = static_cast<__nv_bfloat16*>(a.cache);
  u.n = a.n;
  u.hq = a.hq;
  u.num_rows = a.num_rows;
  u.max_len = a.max_len;
  u.block_table = a.block_table;
  u.block_size = a.block_size;
  u.max_blocks = a.max_blocks;
  u.n_blocks = a.n_blocks;
  u.hkv = 1;
  u.err = a.err;
  const long long warps = static_cast<long long>(a.n) * (1 + (a.q ? a.hq : 0));
  const long long blocks = (warps * 32 + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_dependent(mla_update_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, u);
}

cudaError_t launch_mla_decode(const MlaArgs& a, const MlaPlan& plan, void* workspace, cudaStream_t stream) {
  using namespace mla;
  if (a.n_seqs == 0) return cudaSuccess;
  CUtensorMap tmc;
  const uint64_t rows_total = a.block_table ? static_cast<uint64_t>(a.n_blocks) * a.block_size
                                            : static_cast<uint64_t>(a.num_rows) * a.max_len;
  if (!encode_tmap_2d_bf16(&tmc, a.cache, DR, rows_total, DR * 2, 64, BK)) return cudaErrorInvalidValue;
  Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(a.q);
  prm.rows = a.rows;
  prm.positions = a.positions;
  const size_t o_bytes = static_cast<size_t>(a.n_seqs) * a.hq * plan.n_splits * RANK * sizeof(float);
  prm.ws_o = static_cast<float*>(workspace);
  prm.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + ((o_bytes + 255) & ~size_t(255)));
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.hq = a.hq;
  prm.max_len = a.max_len;
  prm.num_rows = a.num_rows;
  prm.window = a.window;
  prm.scale = a.scale;
  prm.chunk = plan.chunk;
  prm.n_splits = plan.n_splits;
  prm.block_table = a.block_table;
  prm.block_size = a.block_size;
  prm.max_blocks = a.max_blocks;
  prm.n_blocks = a.n_blocks;
  prm.hkv = 1;
  prm.err = a.err;
  // ring, barriers and the give-up word (128 B), exchange buffers: partial scores (8 KB), P^T fragments
  // (1 KB), rescale factors (128 B); 1 KB of alignment slack
  const int smem = NST * STAGE_BYTES + 128 + CWARPS * 4 * 32 * 16 + 4 * 32 * 8 + 32 * 4 + 16 + 1024;
  static_assert(NST * STAGE_BYTES + 128 + CWARPS * 4 * 32 * 16 + 4 * 32 * 8 + 32 * 4 + 16 + 1024 <= 227 * 1024,
                "shared memory budget");
  cudaError_t e;
  if (a.hq == 128) {
    e = launch_mla_pair_decode(a, plan, prm.ws_o, prm.ws_ml, stream);
  } else {
    e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);   // per device
    if (e != cudaSuccess) return e;
    dim3 grid(plan.n_splits, (a.hq + HPC - 1) / HPC, a.n_seqs);
    e = launch_dependent(mla_decode_kernel, grid, dim3(THREADS), smem, stream, tmc, prm);
  }
  if (e != cudaSuccess) return e;
  return launch_dependent(mla_merge_kernel, dim3(a.hq, a.n_seqs), dim3(128), 0, stream, prm);
}

}  // namespace da
