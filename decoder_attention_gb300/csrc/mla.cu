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
// features); four compute warps each serve 8 heads over every key of a tile with m16n8k16 bf16 MMAs: scores
// S^T = K Q^T with keys on M and heads on N (the 8 heads' queries held in registers), O^T += V^T P^T with the
// 512 value features on M (32 MMAs per 16 keys, O^T in registers). Each warp writes its heads' partial (max,
// sum, unnormalised output); mla_merge_kernel combines the chunks in a fixed order.
//
// Roofline: a key costs 1152 bytes and H * (576 + 512) * 2 FLOP (278.5 KFLOP at H = 128, 242 FLOP per byte).
// At that intensity the step needs tensor-core rates; this kernel's legacy MMAs reach ~1600 FLOP per clock
// per SM, and each warp re-reads the tile from shared memory, so it runs well below the HBM bound at H = 128.
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
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NST * STAGE_BYTES);   // full[NST], empty[NST]

  const int c = blockIdx.x, hg = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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

  // -------------------------------------------------------------------- consumers: 8 heads per warp
  const int h0 = hg * HPC + warp * HPW;
  const bool active = h0 < prm.hq;
  const int gq = lane >> 2, cq = lane & 3;
  // B operand of S^T (k = feature, n = head): b0 = Q[h0+gq][16kk + 2cq .. +1], b1 = the same at +8
  uint32_t qb[DR / 16][2];
  {
    const __nv_bfloat16* qrow = prm.q + (static_cast<long long>(s) * prm.hq + (active ? h0 + gq : 0)) * DR;
#pragma unroll
    for (int kk = 0; kk < DR / 16; ++kk) {
      qb[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * cq);
      qb[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * cq);
    }
  }
  const float zmul = prm.scale * kLog2e;
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_run[2] = {0.f, 0.f};
  float o[RANK / 16][4];
#pragma unroll
  for (int mt = 0; mt < RANK / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  bool ok = true;
  const int mi = lane >> 3, r8 = lane & 7;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % NST;
    if (!mbar_wait(full_bar(st), (i / NST) & 1, prm.err)) { ok = false; break; }
    const uint32_t sT = sbase + st * STAGE_BYTES;
    for (int slab = 0; slab < BK / 16 && active; ++slab) {
      const int kb = k0 + i * BK + slab * 16;        // first key of the slab
      const int n_valid = k1 - kb;                   // keys of the 16 inside the chunk (may be <= 0)
      if (n_valid <= 0) break;
      const int n_lo = lo - kb;                      // keys of the 16 below the window (paged tiles only)
      // S^T[16 keys x 8 heads]
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      const int kr = slab * 16 + (mi & 1) * 8 + r8;
#pragma unroll
      for (int kk = 0; kk < DR / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(sT + sw_off(kr, kk * 2 + (mi >> 1)), a0, a1, a2, a3);
        mma_16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
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
      for (int mt = 0; mt < RANK / 16; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
      // P^T as the B operand (k = key, n = head)
      const uint32_t b0 = movmatrix_t(pack2(p0, p1));
      const uint32_t b1 = movmatrix_t(pack2(p2, p3));
      // O^T[512 x 8 heads] += V^T[512 x 16 keys] P^T
      const int vr = slab * 16 + (mi >> 1) * 8 + r8;
      const bool partial = n_valid < 16 || n_lo > 0;
      auto in = [&](int k) { return k >= n_lo && k < n_valid; };
      const uint32_t keep01 = (in(2 * cq) ? 0x0000ffffu : 0u) | (in(2 * cq + 1) ? 0xffff0000u : 0u);
      const uint32_t keep23 = (in(2 * cq + 8) ? 0x0000ffffu : 0u) | (in(2 * cq + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int mt = 0; mt < RANK / 16; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(sT + sw_off(vr, mt * 2 + (mi & 1)), a0, a1, a2, a3);
        if (partial) {   // slots outside the chunk may hold anything (even NaN): 0 * NaN must not reach O
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
  if (!ok || !active) return;
  // row sums: the 8 lanes sharing cq hold disjoint keys
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
  }
  // o[mt][0..1]: feature mt*16 + gq, heads 2cq, 2cq+1; o[mt][2..3]: feature + 8
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int h = h0 + 2 * cq + j;
    const long long slot = (static_cast<long long>(s) * prm.hq + h) * prm.n_splits + c;
    float* wo = prm.ws_o + slot * RANK;
#pragma unroll
    for (int mt = 0; mt < RANK / 16; ++mt) {
      wo[mt * 16 + gq] = o[mt][j];
      wo[mt * 16 + gq + 8] = o[mt][2 + j];
    }
    if (gq == 0) prm.ws_ml[slot] = make_float2(m_run[j], l_run[j]);
  }
}

// One block of 128 threads per (query head, sequence): combine the chunks in order, 4 features a thread.
__global__ void __launch_bounds__(128) mla_merge_kernel(const Params prm) {
  const int h = blockIdx.x, s = blockIdx.y;
  __nv_bfloat16* out = prm.out + (static_cast<long long>(s) * prm.hq + h) * RANK;
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
  mla_update_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(u);
  return cudaGetLastError();
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
  const int smem = NST * STAGE_BYTES + 2 * NST * 8 + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(plan.n_splits, (a.hq + HPC - 1) / HPC, a.n_seqs);
  mla_decode_kernel<<<grid, THREADS, smem, stream>>>(tmc, prm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_merge_kernel<<<dim3(a.hq, a.n_seqs), 128, 0, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace da
