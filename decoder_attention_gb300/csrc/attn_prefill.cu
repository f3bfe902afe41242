// Prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16 operands, fp32 softmax.
//
// Computes causal_attention of DecoderAttention.forward for prefill chunks (page "42. More models: a
// registry, scaled RoPE, sliding windows and latent attention", sections "What differs between model
// families" and "Sliding windows"; soft-capping as "Model resolution" lists it for Gemma 2): for every
// query row, softmax over its visible keys of scale * q.k (optionally c * tanh(. / c)), times V.
//
// CTA = 256 query rows (two 128-row tiles Q0, Q1) of one (sequence, query head). Key tiles of 128 keys
// stream through a 2-stage shared-memory ring by TMA (128-byte swizzle). Roles:
//   warp 8      TMA producer (Q once, then K and V tiles)
//   warp 9      MMA issuer: S_w = Q_w K^T into TMEM, then O_w += P_w V with P_w read from TMEM
//   warps 10-11 idle (they complete the third warpgroup, which setmaxnreg works on)
//   warps 0-3   softmax of Q0 rows, warps 4-7 softmax of Q1 rows: one thread per row; S row from TMEM,
//               mask (only on tiles that need it), online softmax in fp32 (log2 domain, rescale of O
//               only when the running max grows by more than 2^8), P written back into TMEM as bf16
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512). Key tiles outside every query's
// causal window are never loaded (the loop starts at the first tile inside the oldest query's window),
// so a windowed layer costs O(w) per query. Every mbarrier wait is bounded; a wait that gives up sets
// the device error word and the CTA drains and exits.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"

namespace da {
namespace pf {

constexpr int BM = 128;             // rows per Q tile
constexpr int BN = 128;             // keys per K/V tile
constexpr int D = 128;
constexpr int NQT = 2;              // Q tiles per CTA
constexpr int NST = 2;              // K/V ring stages
constexpr int THREADS = 384;     // 3 warpgroups: softmax Q0, softmax Q1, producer/MMA
// setmaxnreg split: launched at 168 per thread (384 x 168 = 64512); softmax warpgroups rise to 224 and
// the producer/MMA warpgroup drops to 56: 256 x 224 + 128 x 56 = 64512, the launch total.
constexpr int REGS_SOFTMAX = 224;
constexpr int REGS_CTRL = 56;
constexpr int HALF = 128 * 128;     // bytes of a 64-wide half of a 128-row tile (16 KB)
constexpr int TILE = 2 * HALF;      // 32 KB
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + NQT * TILE;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_BAR = OFF_V + NST * TILE;
constexpr int N_BARS = 1 + 3 * NST + 2 * NQT + 1;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + TMEM address slot + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: stale max allowed to lag by up to x256

struct Params {
  const int32_t* q_start;
  const int32_t* rows;
  const int32_t* first_pos;
  __nv_bfloat16* out;
  int hq, hkv, max_len, num_rows, window;
  float softcap, scale;
  int* err;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

struct TileInfo {
  int valid[NQT];      // Q tile has at least one real row
  int pmin[NQT], pmax[NQT];
  int tb[NQT], te[NQT];
  int tbeg, tend;
  __device__ bool active(int w, int t) const { return valid[w] && t >= tb[w] && t <= te[w]; }
};

__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmq,
                                                             const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const Params prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x % prm.hq;
  const int s = blockIdx.x / prm.hq;
  const int qt = gridDim.y - 1 - blockIdx.y;      // the longest (latest) query tiles are scheduled first
  const int t0 = prm.q_start[s];
  const int n_b = prm.q_start[s + 1] - t0;
  const int q0 = qt * (NQT * BM);
  if (q0 >= n_b) return;
  const int row = prm.rows[s];
  const int fp = prm.first_pos[s];
  const int kv_len = fp + n_b;
  if (row < 0 || row >= prm.num_rows || fp < 0 || kv_len > prm.max_len) {
    if (threadIdx.x == 0) set_error(prm.err, kErrIndex);
    for (int r = threadIdx.x; r < min(NQT * BM, n_b - q0); r += blockDim.x) {
      uint4* o = reinterpret_cast<uint4*>(prm.out + (static_cast<long long>(t0 + q0 + r) * prm.hq + h) * D);
      for (int j = 0; j < D / 8; ++j) o[j] = make_uint4(0, 0, 0, 0);
    }
    return;
  }
  const int g = h / (prm.hq / prm.hkv);
  const int window = prm.window;

  TileInfo ti;
#pragma unroll
  for (int w = 0; w < NQT; ++w) {
    const int r0 = q0 + w * BM;
    ti.valid[w] = r0 < n_b;
    const int nr = ti.valid[w] ? min(BM, n_b - r0) : 1;
    ti.pmin[w] = fp + r0;
    ti.pmax[w] = fp + r0 + nr - 1;
    const int lo = window > 0 ? max(0, ti.pmin[w] - window + 1) : 0;
    ti.tb[w] = lo / BN;
    ti.te[w] = ti.pmax[w] / BN;
  }
  ti.tbeg = ti.tb[0];
  ti.tend = ti.valid[1] ? ti.te[1] : ti.te[0];
  const int n_tiles = ti.tend - ti.tbeg + 1;

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + OFF_BAR;
  const uint32_t bar_q = bar;
  auto bar_kfull = [&](int st) { return bar + 8u * (1 + st); };
  auto bar_vfull = [&](int st) { return bar + 8u * (1 + NST + st); };
  auto bar_empty = [&](int st) { return bar + 8u * (1 + 2 * NST + st); };
  auto bar_sfull = [&](int w) { return bar + 8u * (1 + 3 * NST + w); };
  auto bar_pfull = [&](int w) { return bar + 8u * (1 + 3 * NST + NQT + w); };
  const uint32_t bar_odone = bar + 8u * (1 + 3 * NST + 2 * NQT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + N_BARS * 8);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar_q, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar_kfull(i), 1);
      mbar_init(bar_vfull(i), 1);
      mbar_init(bar_empty(i), 1);
    }
    for (int w = 0; w < NQT; ++w) {
      mbar_init(bar_sfull(w), 1);
      mbar_init(bar_pfull(w), BM);
    }
    mbar_init(bar_odone, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int* vabort = &abort_flag;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
    if (warp == 8 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      const int nq = ti.valid[1] ? 2 : 1;
      mbar_arrive_expect_tx(bar_q, nq * TILE);
      for (int w = 0; w < nq; ++w) {
        const int tok = t0 + q0 + w * BM;
        tma_load_3d(sbase + OFF_Q + w * TILE, &tmq, bar_q, 0, h, tok);
        tma_load_3d(sbase + OFF_Q + w * TILE + HALF, &tmq, bar_q, 64, h, tok);
      }
      const int plane = (row * prm.hkv + g) * prm.max_len;
      int issued = 0;
      for (int i = 0; i < n_tiles && !*vabort; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(bar_empty(st), ((i / NST) + 1) & 1, prm.err)) {
          abort_flag = 1;
          break;
        }
        const int key = plane + (ti.tbeg + i) * BN;
        mbar_arrive_expect_tx(bar_kfull(st), TILE);
        tma_load_2d(sbase + OFF_K + st * TILE, &tmk, bar_kfull(st), 0, key);
        tma_load_2d(sbase + OFF_K + st * TILE + HALF, &tmk, bar_kfull(st), 64, key);
        mbar_arrive_expect_tx(bar_vfull(st), TILE);
        tma_load_2d(sbase + OFF_V + st * TILE, &tmv, bar_vfull(st), 0, key);
        tma_load_2d(sbase + OFF_V + st * TILE + HALF, &tmv, bar_vfull(st), 64, key);
        ++issued;
      }
      // every issued copy must land before the CTA's shared memory is released
      mbar_wait(bar_q, 0, prm.err);
      for (int i = max(0, issued - NST); i < issued; ++i) {
        mbar_wait(bar_kfull(i % NST), (i / NST) & 1, prm.err);
        mbar_wait(bar_vfull(i % NST), (i / NST) & 1, prm.err);
      }
    } else if (warp == 9 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);   // Q, K both K-major
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);     // P (TMEM), V MN-major
      int nact[NQT] = {0, 0};
      bool ok = mbar_wait(bar_q, 0, prm.err);
      tc_fence_after();
      for (int i = 0; ok && i < n_tiles; ++i) {
        if (*vabort) break;
        const int t = ti.tbeg + i;
        const int st = i % NST;
        const uint32_t ph = (i / NST) & 1;
        if (!mbar_wait(bar_kfull(st), ph, prm.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = sbase + OFF_K + st * TILE;
        const bool act[NQT] = {ti.active(0, t), ti.active(1, t)};
#pragma unroll
        for (int w = 0; w < NQT; ++w) {
          if (!act[w]) continue;
          const uint32_t qb = sbase + OFF_Q + w * TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;
            mma_ss(tmem + w * BN, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), idesc_qk,
                   kk > 0 ? 1u : 0u);
          }
          tc_commit(bar_sfull(w));
        }
        if (!mbar_wait(bar_vfull(st), ph, prm.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t vb = sbase + OFF_V + st * TILE;
#pragma unroll
        for (int w = 0; w < NQT; ++w) {
          if (!act[w] || !ok) continue;
          if (!mbar_wait(bar_pfull(w), nact[w] & 1, prm.err)) {
            ok = false;
            continue;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            mma_ts(tmem + 256 + w * D, tmem + w * BN + kk * 8, sdesc_sw128(vb + kk * 2048, HALF, 1024), idesc_pv,
                   (nact[w] > 0 || kk > 0) ? 1u : 0u);
          }
          ++nact[w];
        }
        tc_commit(bar_empty(st));
      }
      if (!ok) abort_flag = 1;
      tc_commit(bar_odone);
      mbar_wait(bar_odone, 0, prm.err);   // all MMAs done before TMEM may be released
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
    // ---------------------------------------------------------------- softmax (8 warps, 1 row each thread)
    const int w = warp >> 2;             // which Q tile
    const int wi = warp & 3;             // TMEM lane quarter
    const int r = wi * 32 + lane;        // row within the tile
    const int qrow = q0 + w * BM + r;    // row within the chunk
    const bool row_ok = qrow < n_b;
    const int p = fp + qrow;
    const uint32_t lane_addr = static_cast<uint32_t>(wi * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + w * BN;
    const uint32_t t_o = tmem + lane_addr + 256 + w * D;
    const float cap = prm.softcap;
    const float zmul = cap > 0.f ? prm.scale / cap : prm.scale * kLog2e;
    const float cap_l2 = cap * kLog2e;
    const bool my_valid = w == 0 ? ti.valid[0] : ti.valid[1];
    const int my_tb = w == 0 ? ti.tb[0] : ti.tb[1];
    const int my_te = w == 0 ? ti.te[0] : ti.te[1];
    const int my_pmin = w == 0 ? ti.pmin[0] : ti.pmin[1];
    const int my_pmax = w == 0 ? ti.pmax[0] : ti.pmax[1];
    float m = -CUDART_INF_F, l = 0.f;
    int nact = 0;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int t = ti.tbeg + i;
      if (!my_valid || t < my_tb || t > my_te) continue;
      // outcomes are made warp-uniform: the TMEM loads and stores below are warp-collective
      if (__any_sync(0xffffffffu, *vabort != 0)) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull(w), nact & 1, prm.err))) {
        abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t zr[BN];
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) tmem_ld32(t_s + j * 32, *reinterpret_cast<uint32_t(*)[32]>(&zr[j * 32]));
      tmem_wait_ld();
      const int kstart = t * BN;
      const bool need_mask = !(kstart + BN - 1 <= my_pmin &&
                               (window == 0 || my_pmax - kstart <= window - 1) && kstart + BN <= kv_len);
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        float v = __uint_as_float(zr[c]) * zmul;
        if (cap > 0.f) v = cap_l2 * tanh_fast(v);
        if (need_mask) {
          const int j = kstart + c;
          const bool vis = j <= p && (window == 0 || p - j <= window - 1) && j < kv_len;
          v = vis ? v : -CUDART_INF_F;
        }
        zr[c] = __float_as_uint(v);
        tmax = fmaxf(tmax, v);
      }
      const float m_new = fmaxf(m, tmax);
      const bool grow = m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m - m_new);   // 0 when m was -inf
        l *= alpha;
        m = m_new;
      }
      if (nact > 0 && __any_sync(0xffffffffu, grow)) {
        // O row *= alpha (rows that did not grow multiply by 1). PV of the previous tile has completed:
        // its commit preceded the S commit just waited on.
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          uint32_t ov[32];
          tmem_ld32(t_o + j * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(t_o + j * 32, ov);
        }
      }
      const float mu = (m == -CUDART_INF_F) ? 0.f : m;
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float pa = ex2(__uint_as_float(zr[j * 32 + 2 * e]) - mu);
          const float pb = ex2(__uint_as_float(zr[j * 32 + 2 * e + 1]) - mu);
          l += pa + pb;
          pk[e] = pack_bf16(pa, pb);
        }
        tmem_st16(t_s + j * 16, pk);     // P (bf16, 2 per column) over the first half of the S columns
      }
      tmem_wait_st();
      if (kstart + BN > kv_len) {
        // V rows past the row's last key hold whatever the cache holds there (maybe NaN); P is 0 there,
        // but 0 * NaN is NaN, so zero those rows before the tensor core reads them (after the V copy has
        // landed; the stage cannot be refilled before this tile's PV, which waits for us).
        if (!__all_sync(0xffffffffu, mbar_wait(bar_vfull(i % NST), (i / NST) & 1, prm.err))) {
          abort_flag = 1;
          ok = false;
          break;
        }
        if (kstart + r >= kv_len) {
          uint4* vrow0 = reinterpret_cast<uint4*>(smem + OFF_V + (i % NST) * TILE + r * 128);
          uint4* vrow1 = reinterpret_cast<uint4*>(smem + OFF_V + (i % NST) * TILE + HALF + r * 128);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            vrow0[e] = make_uint4(0, 0, 0, 0);
            vrow1[e] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(bar_pfull(w));
      ++nact;
    }
    // ------------------------------------------------------------ epilogue: O / l -> out
    if (ok && __all_sync(0xffffffffu, mbar_wait(bar_odone, 0, prm.err))) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(prm.out + (static_cast<long long>(t0 + qrow) * prm.hq + h) * D);
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        uint32_t ov[32];
        tmem_ld32(t_o + j * 32, ov);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 u;
            u.x = pack_bf16(__uint_as_float(ov[8 * e + 0]) * inv_l, __uint_as_float(ov[8 * e + 1]) * inv_l);
            u.y = pack_bf16(__uint_as_float(ov[8 * e + 2]) * inv_l, __uint_as_float(ov[8 * e + 3]) * inv_l);
            u.z = pack_bf16(__uint_as_float(ov[8 * e + 4]) * inv_l, __uint_as_float(ov[8 * e + 5]) * inv_l);
            u.w = pack_bf16(__uint_as_float(ov[8 * e + 6]) * inv_l, __uint_as_float(ov[8 * e + 7]) * inv_l);
            orow[j * 4 + e] = u;
          }
        }
      }
    } else {
      abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace pf

cudaError_t launch_prefill_bf16(const AttnArgs& a, cudaStream_t stream) {
  using namespace pf;
  if (a.n_seqs == 0 || a.max_q_len == 0 || a.n_tokens == 0) return cudaSuccess;
  CUtensorMap tmq, tmk, tmv;
  const uint64_t rows_total = static_cast<uint64_t>(a.num_rows) * a.hkv * a.max_len;
  // q_rot [N, Hq, D]: rows past N are zero-filled by the copy engine, never read from memory
  const uint64_t n_tok = static_cast<uint64_t>(a.n_tokens);
  if (!encode_tmap_3d_bf16(&tmq, a.q_rot, D, a.hq, n_tok, D * 2, static_cast<uint64_t>(a.hq) * D * 2, 64, 1, BM) ||
      !encode_tmap_2d_bf16(&tmk, a.k_cache, D, rows_total, D * 2, 64, BN) ||
      !encode_tmap_2d_bf16(&tmv, a.v_cache, D, rows_total, D * 2, 64, BN))
    return cudaErrorInvalidValue;
  Params prm;
  prm.q_start = a.q_start;
  prm.rows = a.rows;
  prm.first_pos = a.first_pos;
  prm.out = static_cast<__nv_bfloat16*>(a.out);
  prm.hq = a.hq;
  prm.hkv = a.hkv;
  prm.max_len = a.max_len;
  prm.num_rows = a.num_rows;
  prm.window = a.window;
  prm.softcap = a.softcap;
  prm.scale = a.scale;
  prm.err = a.err;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int n_qt = (a.max_q_len + NQT * BM - 1) / (NQT * BM);
  dim3 grid(a.hq * a.n_seqs, n_qt);
  prefill_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(tmq, tmk, tmv, prm);
  return cudaGetLastError();
}

}  // namespace da
