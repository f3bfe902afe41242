// The projections on either side of the attention step on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", DecoderAttention:
// q = q_proj(x), k = k_proj(x), v = v_proj(x), then q_norm/k_norm, apply_rope and cache.update; after
// attention, o_proj. Both are a GEMM Y = X W^T (+ b) with X [M, K] and W [N, K] bf16, fp32 accumulation.
//
// gemm_kernel<EPI> runs persistent clusters of two CTAs (one per SM) over 256 x 256 output tiles. CTA r of a
// pair stages, per 64-wide K slice, X rows r*128.. of the tile and W rows r*128.. (its half of the tile's
// columns) through a 6-stage ring (128-byte swizzle); one thread of CTA 0 issues tcgen05.mma with
// cta_group::2 (M 256, N 256, K 16), which reads both CTAs' slices and leaves rows r*128.. of the tile in CTA
// r's TMEM, in one of two 256-column accumulators. Per SM this moves half the operand bytes of a one-CTA
// 128 x 256 tile through shared memory (each W column slice is staged once per pair, not per CTA), which is
// what keeps the tensor pipe fed. A warpgroup of 128 epilogue threads per CTA (one output row each) drains
// the other accumulator meanwhile:
//   EPI_QKV   the tile is two 128-wide heads of the stacked q/k/v projection. Per token and head: bias, then
//             for q and k the per-head RMSNorm (when the layer has norm weights) and the split-half RoPE with
//             the token's cos/sin, rounded to bf16 and written to q_rot or the token's cache slot (k); v heads
//             go to their cache slot unchanged. The q/k/v intermediate never reaches memory.
//   EPI_PLAIN Y (+ b) rounded to bf16 (o_proj).
// Every wait is bounded; a wait that gives up sets the device error word and the CTA drains and exits.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {
namespace proj {

constexpr int BM = 128, BN = 256, BK = 64;     // per CTA: 128 rows of the pair's 256-row tile, all 256 columns
constexpr int CLUSTER = 2;
constexpr int NS = 6;                          // ring stages
constexpr int A_BYTES = BM * BK * 2;           // 16 KB: this CTA's X rows
constexpr int B_BYTES = (BN / 2) * BK * 2;     // 16 KB: this CTA's half of the W rows
constexpr int STAGE = A_BYTES + B_BYTES;       // 32 KB
constexpr int THREADS = 256;                   // warp 0 TMA, warp 1 MMA (CTA 0), warp 2 TMEM owner, warps 4-7 epilogue
constexpr int EPI_QKV = 0, EPI_PLAIN = 1;
// barriers: full[NS] (CTA 0's count the pair's bytes), empty[NS], acc_full[2], acc_empty[2] (CTA 0's count the
// pair's eight epilogue warps)
constexpr int B_FU = 0, B_EM = NS, B_AF = 2 * NS, B_AE = 2 * NS + 2, N_BARS = 2 * NS + 4;
constexpr int SMEM_BYTES = NS * STAGE + 256 + 1024;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

struct Params {
  int m, n, k;                     // Y [m, n] = X [m, k] W [n, k]^T
  const float* bias;               // [n] or NULL
  __nv_bfloat16* y;                // EPI_PLAIN: [m, n]
  // EPI_QKV
  int hq, hkv;                     // heads (d = 128, all 128 dims rotated)
  const float* q_norm_w;           // [128] or NULL
  const float* k_norm_w;
  float eps;
  const float* cos;                // [m, 64]
  const float* sin;
  const int32_t* rows;             // [m]
  const int32_t* positions;        // [m]
  __nv_bfloat16* q_rot;            // [m, hq, 128]
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int num_rows, max_len;
  const int32_t* block_table;      // paged pool or NULL
  int block_size, max_blocks, n_blocks;
  int* err;
};

template <int EPI>
__global__ void __cluster_dims__(CLUSTER, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + NS * STAGE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + NS * STAGE + N_BARS * 8);
  auto B = [&](int i) { return bar + 8u * i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a work item is one n-tile of a pair of m-tiles; CTA `rank` of the cluster takes m-tile 2 * pair + rank
  // (past the last m-tile it computes on the zeros TMA fills in and stores nothing)
  const int rank = static_cast<int>(cluster_rank());
  const int m_tiles = (prm.m + BM - 1) / BM, n_tiles = prm.n / BN;
  const int cid = blockIdx.x / CLUSTER, n_clusters = gridDim.x / CLUSTER;
  const int n_work = ((m_tiles + 1) / 2) * n_tiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(B(B_FU + i), 1);
      mbar_init(B(B_EM + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B(B_AF + i), 1);
      mbar_init(B(B_AE + i), 4 * CLUSTER);   // one arrival per epilogue warp of the pair
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers are initialised before any copy, commit or arrival reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kb_n = prm.k / BK;
  pdl_wait();   // inputs written by the stream's previous kernel are visible

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    prefetch_tmap(&tma);
    prefetch_tmap(&tmb);
    const uint32_t full0 = map_to_rank(B(B_FU), 0);   // the pair's full barriers live in CTA 0
    int it = 0;
    bool ok = true;
    for (int w = cid; ok && w < n_work; w += n_clusters) {
      const int nt = w % n_tiles, mt = 2 * (w / n_tiles) + rank;   // W (all n-tiles) stays in L2; X read once
      for (int kb = 0; kb < kb_n; ++kb, ++it) {
        const int s = it % NS;
        if (it >= NS && !mbar_wait(B(B_EM + s), ((it / NS) - 1) & 1, prm.err)) { ok = false; break; }
        const uint32_t dst = sbase + s * STAGE;
        if (rank == 0) mbar_arrive_expect_tx(B(B_FU + s), CLUSTER * STAGE);   // both CTAs' slices
        tma_load_2d_pair(dst, &tma, full0 + 8u * s, kb * BK, mt * BM);
        tma_load_2d_pair(dst + A_BYTES, &tmb, full0 + 8u * s, kb * BK, nt * BN + rank * (BN / 2));
      }
    }
    // the last stages are released: the pair's MMAs have read every slice this CTA staged
    for (int j = max(0, it - NS); j < it; ++j) mbar_wait(B(B_EM + j % NS), (j / NS) & 1, prm.err);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------------------------------------------------------- MMA issuer (CTA 0 for the pair)
    constexpr uint32_t idesc = idesc_bf16_f32(CLUSTER * BM, BN, false, false);
    int it = 0, tcount = 0;
    bool ok = true;
    for (int w = cid; ok && w < n_work; w += n_clusters, ++tcount) {
      const int buf = tcount & 1;
      if (tcount >= 2 && !mbar_wait_cluster(B(B_AE + buf), ((tcount >> 1) - 1) & 1, prm.err)) break;   // drained
      tc_fence_after();
      const uint32_t d = tmem + buf * BN;
      for (int kb = 0; kb < kb_n; ++kb, ++it) {
        const int s = it % NS;
        if (!mbar_wait(B(B_FU + s), (it / NS) & 1, prm.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a = sbase + s * STAGE, b = a + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss_pair(d, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(b + kk * 32, 16, 1024), idesc,
                      (kb | kk) != 0);
        tc_commit_pair(B(B_EM + s));   // the stage is free in both CTAs once these MMAs have read it
      }
      if (ok) tc_commit_pair(B(B_AF + buf));
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue: one output row per thread
    const int q4 = warp - 4;                 // TMEM lane quarter
    const int r = q4 * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    const KvLayout kvl = kv_layout(prm);
    const uint32_t acc_empty0 = map_to_rank(B(B_AE), 0);
    int tcount = 0;
    for (int w = cid; w < n_work; w += n_clusters, ++tcount) {
      const int buf = tcount & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(B(B_AF + buf), (tcount >> 1) & 1, prm.err))) break;
      tc_fence_after();
      const int nt = w % n_tiles, mt = 2 * (w / n_tiles) + rank;
      const int row = mt * BM + r;           // output row (token)
      const bool live = row < prm.m;
#pragma unroll 1
      for (int half = 0; half < BN / 128; ++half) {
        const int col0 = nt * BN + half * 128;
        float x[128];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_addr + buf * BN + half * 128 + j * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) x[j * 32 + e] = __uint_as_float(v[e]);
        }
        if (!live) continue;
        if (prm.bias) {
          const float4* b4 = reinterpret_cast<const float4*>(prm.bias + col0);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float4 b = b4[e];
            x[4 * e] += b.x;
            x[4 * e + 1] += b.y;
            x[4 * e + 2] += b.z;
            x[4 * e + 3] += b.w;
          }
        }
        __nv_bfloat16* dst;
        if constexpr (EPI == EPI_PLAIN) {
          dst = prm.y + static_cast<long long>(row) * prm.n + col0;
        } else {
          const int head = col0 / 128;                       // stacked: q heads, then k heads, then v heads
          const bool is_q = head < prm.hq, is_k = !is_q && head < prm.hq + prm.hkv;
          if (is_q || is_k) {
            const float* nw = is_q ? prm.q_norm_w : prm.k_norm_w;
            if (nw) {
              float ss = 0.f;
#pragma unroll
              for (int e = 0; e < 128; ++e) ss += x[e] * x[e];
              const float inv = rsqrtf(ss * (1.f / 128.f) + prm.eps);
              const float4* w4 = reinterpret_cast<const float4*>(nw);
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float4 wv = w4[e];
                x[4 * e] *= inv * wv.x;
                x[4 * e + 1] *= inv * wv.y;
                x[4 * e + 2] *= inv * wv.z;
                x[4 * e + 3] *= inv * wv.w;
              }
            }
            const float4* cs = reinterpret_cast<const float4*>(prm.cos + static_cast<long long>(row) * 64);
            const float4* sn = reinterpret_cast<const float4*>(prm.sin + static_cast<long long>(row) * 64);
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4) {   // split-half pairs (i, i + 64), four at a time
              const float4 c4 = cs[i4], s4 = sn[i4];
              const float cv[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int i = 4 * i4 + j;
                const float a = x[i], b = x[i + 64];
                x[i] = a * cv[j] - b * sv[j];
                x[i + 64] = b * cv[j] + a * sv[j];
              }
            }
          }
          if (is_q) {
            dst = prm.q_rot + (static_cast<long long>(row) * prm.hq + head) * 128;
          } else {
            const int g = is_k ? head - prm.hq : head - prm.hq - prm.hkv;
            const long long slot = kv_slot(kvl, prm.rows[row], prm.positions[row]);
            if (slot < 0) {
              set_error(prm.err, kErrIndex);
              continue;
            }
            dst = (is_k ? prm.k_cache : prm.v_cache) + (slot + g * kv_head_stride(kvl)) * 128;
          }
        }
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int c8 = 0; c8 < 16; ++c8) {
          uint4 pk;
          pk.x = pack_bf16x2(x[c8 * 8 + 0], x[c8 * 8 + 1]);
          pk.y = pack_bf16x2(x[c8 * 8 + 2], x[c8 * 8 + 3]);
          pk.z = pack_bf16x2(x[c8 * 8 + 4], x[c8 * 8 + 5]);
          pk.w = pack_bf16x2(x[c8 * 8 + 6], x[c8 * 8 + 7]);
          d4[c8] = pk;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * buf);   // this warp's accumulator lanes are drained
    }
  }
  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while a copy, commit or arrival of the pair may still target its shared memory or TMEM:
  // both epilogues have seen the last accumulators, so every MMA and copy of the pair has completed
  cluster_sync();
  tc_fence_after();
  if (warp == 2) tmem_dealloc_pair(tmem, 512);
}

}  // namespace proj

cudaError_t launch_proj(const ProjArgs& a, cudaStream_t stream) {
  using namespace proj;
  if (a.m == 0) return cudaSuccess;
  CUtensorMap tma, tmb;
  if (!encode_tmap_2d_bf16(&tma, a.x, a.k, a.m, static_cast<uint64_t>(a.k) * 2, BK, BM) ||
      !encode_tmap_2d_bf16(&tmb, a.w, a.k, a.n, static_cast<uint64_t>(a.k) * 2, BK, BN / 2))
    return cudaErrorInvalidValue;
  Params p;
  p.m = a.m;
  p.n = a.n;
  p.k = a.k;
  p.bias = a.bias;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.q_norm_w = a.q_norm_w;
  p.k_norm_w = a.k_norm_w;
  p.eps = a.eps;
  p.cos = a.cos;
  p.sin = a.sin;
  p.rows = a.rows;
  p.positions = a.positions;
  p.q_rot = static_cast<__nv_bfloat16*>(a.q_rot);
  p.k_cache = static_cast<__nv_bfloat16*>(a.k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(a.v_cache);
  p.num_rows = a.num_rows;
  p.max_len = a.max_len;
  p.block_table = a.block_table;
  p.block_size = a.block_size;
  p.max_blocks = a.max_blocks;
  p.n_blocks = a.n_blocks;
  p.err = a.err;
  const bool qkv = a.q_rot != nullptr;
  cudaError_t e = cudaFuncSetAttribute(qkv ? gemm_kernel<EPI_QKV> : gemm_kernel<EPI_PLAIN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // persistent clusters: as many as can be resident at once (a GPC with an odd number of free SMs leaves one idle)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm / CLUSTER * CLUSTER);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  int resident = 0;
  e = cudaOccupancyMaxActiveClusters(&resident, qkv ? gemm_kernel<EPI_QKV> : gemm_kernel<EPI_PLAIN>, &cfg);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  const long long work = static_cast<long long>(((a.m + BM - 1) / BM + 1) / 2) * (a.n / BN);   // tile pairs
  cfg.gridDim = dim3(CLUSTER * static_cast<unsigned>(std::min<long long>(work, resident)));
  // programmatic dependent launch: the kernel may start while the stream's previous kernel finishes (it waits
  // in pdl_wait before touching memory)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return qkv ? cudaLaunchKernelEx(&cfg, gemm_kernel<EPI_QKV>, tma, tmb, p)
             : cudaLaunchKernelEx(&cfg, gemm_kernel<EPI_PLAIN>, tma, tmb, p);
}

}  // namespace da
