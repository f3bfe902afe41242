// MLA decode with absorbed up-projections on the sm_103a tensor cores, for layers with 128 query heads
// (DeepSeek-V2/V3): bf16 rows of 576 (latent 512, rotary 64), one query token per sequence.
//
// Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", sections "Multi-head
// latent attention" and "Serving it: absorbing the up-projections": decode is multi-query attention of every
// head's latent query (q = [W_uk^T q_nope, q_rope]) against the cached rows, whose first 512 features are the
// values; the output is the latent per head (W_uv is applied outside). The arithmetic is the same as the
// legacy-MMA kernel in mla.cu; only the tiling differs.
//
// mla_pair_kernel: a cluster of two CTAs per (key chunk, sequence) walks the chunk in tiles of 256 keys.
//   Scores, transposed:  S^T = K Q^T, one cta_group::2 MMA chain (M 256 keys, N 128 heads, K 576): CTA r
//     stages its 128 keys of the tile (all 576 features) and query heads [64 r, 64 r + 64), and gets the
//     scores of its keys for all 128 heads in TMEM (lane = key, column = head).
//   Output, transposed:  O^T += V^T P^T, one cta_group::2 MMA chain per 256 value features (M 256 features,
//     N 128 heads, K 256 keys): CTA r stages value features [256 fb + 128 r, +128) of all 256 keys and the
//     probabilities of heads [64 r, 64 r + 64), and accumulates its 2 x 128 features for all heads in TMEM.
//   So every score and output element is computed once, both MMAs run at M 256 N 128, and each CTA moves half
//   of the tile's bytes. Between the two, four warps per CTA (one TMEM lane quarter each) run the online
//   softmax over the keys (per head = per TMEM column, reduced across lanes by shuffles), the two CTAs trade
//   their per-head tile maxima (128 floats) and each writes the probabilities of the other CTA's heads straight
//   into its shared memory. The running max moves only when it grows by more than 2^8 (both CTAs decide
//   alike, from the same numbers), so O^T is rescaled in TMEM on few tiles.
// Per pair: TMEM 2 x 128 columns of scores (double-buffered) + 2 x 128 of output; shared memory 72 KB of
// queries, a 3-slot ring of 32 KB (128 keys x 128 features), 32 KB of P^T.
// The chunk's partials (max, sum, unnormalised output per head) go to the same workspace the legacy kernel
// uses, and mla_merge_kernel combines the chunks. Every wait is bounded; a wait that gives up sets the error
// word, and the CTA skips the remaining waits (finishing in bounded time) and still meets every barrier.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {
namespace mlap {

constexpr int H = 128, HH = 64;              // heads; heads staged per CTA
constexpr int DR = 576;                      // a cached row: latent 512 + rotary 64
constexpr int TK = 128, PT = 256;            // keys per CTA, per pair tile
constexpr int BOX = 64 * 128;                // one TMA load: 64 rows x 64 features (128 B, swizzled) = 8 KB
constexpr int ATOM = 2 * BOX;                // 128 rows x 64 features = 16 KB
constexpr int SLOT = 2 * ATOM;               // 128 rows x 128 features = 32 KB
constexpr int NSLOT = 3;
constexpr int Q_OFF = 0, Q_BYTES = 9 * BOX;  // 9 boxes of 64 heads x 64 features
constexpr int RING_OFF = Q_OFF + Q_BYTES;
constexpr int PT_OFF = RING_OFF + NSLOT * SLOT;   // P^T: [256 keys][64 heads] bf16, 128-byte swizzle
constexpr int MX_OFF = PT_OFF + PT * 128;         // peer's tile maxima [2][128] f32
constexpr int WM_OFF = MX_OFF + 2 * H * 4;        // per-warp column maxima / sums [4][128] f32
constexpr int M_OFF = WM_OFF + 4 * H * 4;         // running max per head (log2 units)
constexpr int AL_OFF = M_OFF + H * 4;             // rescale factor per head
constexpr int LP_OFF = AL_OFF + H * 4;            // CTA 1's sums per head (received by CTA 0)
constexpr int FILL_OFF = LP_OFF + H * 4;           // boundary group: [2][4] int (destination, first key)
constexpr int BAR_OFF = FILL_OFF + 2 * 4 * 4;
// barriers: full[NSLOT] (CTA 0's count the pair's bytes), empty[NSLOT], s_full[2], s_free[2], p_full, o_done,
// mx_full[2], q_full, split[2] (CTA 0's: the hand-filled value rows of the group holding the last visible key
// are in place in both CTAs, one barrier for each of the two value slots that carry it), fill[2] (the producer
// hands such a slot to the filling warp)
constexpr int B_FULL = 0, B_EMPTY = B_FULL + NSLOT, B_SFULL = B_EMPTY + NSLOT, B_SFREE = B_SFULL + 2,
              B_PFULL = B_SFREE + 2, B_ODONE = B_PFULL + 1, B_MXFULL = B_ODONE + 1, B_QFULL = B_MXFULL + 2,
              B_SPLIT = B_QFULL + 1, B_FILL = B_SPLIT + 2, N_BARS = B_FILL + 2;
constexpr int SMEM_BYTES = BAR_OFF + N_BARS * 8 + 8 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
constexpr int THREADS = 384;   // warp 0 TMA, warp 1 MMA (CTA 0), warp 2 TMEM owner, warps 4-11 softmax
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGrow = 8.0f;  // log2 units: the running max may lag the true max by up to x256

struct Params {
  const int32_t* rows;
  const int32_t* positions;
  float* ws_o;                // [S, H, n_splits, 512]
  float2* ws_ml;              // [S, H, n_splits] (max in log2 units, sum)
  int hq, max_len, num_rows, window;
  float scale;
  int chunk, n_splits;
  const int32_t* block_table;
  int block_size, max_blocks, n_blocks;
  int hkv;
  int oob_row;                      // first row past the cache (TMA reads zeros there)
  int* err;
};

__device__ __forceinline__ void bar_sync_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool bar_or_softmax(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Column reduction of a warp's 32 x 32 block (lane = row, x[] = columns): on return lane L holds the
// reduction of column L over the 32 rows. Each halving step trades the half a lane gives away for its
// partner's copy of the half it keeps (31 shuffles in all).
template <bool MAX>
__device__ __forceinline__ float warp_colreduce32(const float (&x)[32], int lane) {
  auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
  float a16[16], a8[8], a4[4], a2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2, u1 = lane & 1;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    a16[i] = op(u16 ? x[i + 16] : x[i], __shfl_xor_sync(0xffffffffu, u16 ? x[i] : x[i + 16], 16));
#pragma unroll
  for (int i = 0; i < 8; ++i)
    a8[i] = op(u8 ? a16[i + 8] : a16[i], __shfl_xor_sync(0xffffffffu, u8 ? a16[i] : a16[i + 8], 8));
#pragma unroll
  for (int i = 0; i < 4; ++i)
    a4[i] = op(u4 ? a8[i + 4] : a8[i], __shfl_xor_sync(0xffffffffu, u4 ? a8[i] : a8[i + 4], 4));
#pragma unroll
  for (int i = 0; i < 2; ++i)
    a2[i] = op(u2 ? a4[i + 2] : a4[i], __shfl_xor_sync(0xffffffffu, u2 ? a4[i] : a4[i + 2], 2));
  return op(u1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, u1 ? a2[0] : a2[1], 1));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The 64-key group starting at key g holds the last visible key p and keys past it, which were never written.
__device__ __forceinline__ bool holds_last(int g, int p) { return g <= p && g + 63 > p; }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmc,
                    const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) { return sb + BAR_OFF + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BAR_OFF + N_BARS * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = static_cast<int>(cluster_rank());
  const int c = blockIdx.x >> 1, s = blockIdx.z;

  pdl_wait();   // the stream's previous kernel (the cache update) has finished writing the cache
  // both CTAs of the pair see the same sequence and chunk, so they leave together
  const int p = prm.positions[s];
  const int row = prm.rows[s];
  if (row < 0 || row >= prm.num_rows || p < 0 || p >= prm.max_len) {
    if (threadIdx.x == 0 && c == 0 && r == 0) set_error(prm.err, kErrIndex);
    return;   // the merge kernel writes zeros for this sequence
  }
  const bool paged = prm.block_table != nullptr;
  const int lo = prm.window > 0 ? max(0, p + 1 - prm.window) : 0;
  const int base = paged ? (lo & ~63) : lo;      // paged: 64-key groups lie in one block
  const int k0 = base + c * prm.chunk;
  if (k0 > p) return;
  const int k1 = min(k0 + prm.chunk, p + 1);
  const int n_tiles = (k1 - k0 + PT - 1) / PT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(bar(B_FULL + i), 1);
      mbar_init(bar(B_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SFREE + i), 16);   // eight softmax warps in each CTA
      mbar_init(bar(B_MXFULL + i), 4);   // the peer's four softmax warps
    }
    mbar_init(bar(B_PFULL), 16);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_SPLIT), 2);        // both CTAs' producer warps
    mbar_init(bar(B_SPLIT + 1), 2);
    mbar_init(bar(B_FILL), 1);
    mbar_init(bar(B_FILL + 1), 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // columns: S^T buffers at 0 and 128, O^T at 256 (fb 0) and 384 (fb 1)

  float m_reg = -CUDART_INF_F, l_cta = 0.f;   // softmax threads: head (threadIdx.x - 128)

  // the 64-key group holding the last visible key p, when it lies in this chunk and holds keys past p (whose
  // value rows were never written): warp 3 fills its two value slots by hand
  const bool has_split = k1 == p + 1 && ((p - k0) & 63) != 63;
  int* fill = reinterpret_cast<int*>(smem + FILL_OFF);
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer (both CTAs)
    // Groups with no visible key, value groups past p and missing blocks are read from past the end of the
    // cache, where TMA fills zeros: no unwritten slot reaches O through 0 * NaN. The value rows of the group
    // holding p go to warp 3 instead (rows up to p copied, the rest zero).
    prefetch_tmap(&tmq);
    prefetch_tmap(&tmc);
    const uint32_t full0 = map_to_rank(bar(B_FULL), 0);
    if (r == 0) mbar_arrive_expect_tx(bar(B_QFULL), 2 * Q_BYTES);
#pragma unroll 1
    for (int b = 0; b < 9; ++b)
      tma_load_2d_pair(sb + Q_OFF + b * BOX, &tmq, map_to_rank(bar(B_QFULL), 0), b * 64, s * H + r * HH);
    const KvLayout kvl = kv_layout(prm);
    const long long plane = static_cast<long long>(row) * prm.max_len;
    // cache rows of the four 64-key groups of tile t (-1: outside the cache or a missing block), looked up once
    // per tile with independent loads and kept for the tile's value slots, which come a tile later
    long long ge[4], go[4];   // even and odd tiles, in registers (selected, never indexed at run time)
    auto lookup = [&](int t) {
      long long v[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int g = k0 + t * PT + m * 64;
        v[m] = paged ? kv_slot(kvl, row, g) : plane + g;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if (t & 1) go[m] = v[m];
        else ge[m] = v[m];
      }
    };
    auto group_row = [&](int t, int m, bool is_v) -> int {
      const int g = k0 + t * PT + m * 64;
      if (g + 63 < lo || (is_v && g > p)) return prm.oob_row;
      const long long* gs = (t & 1) ? go : ge;
      const long long sl = m == 0 ? gs[0] : m == 1 ? gs[1] : m == 2 ? gs[2] : gs[3];
      if (sl < 0) {
        if (g <= p) set_error(prm.err, kErrIndex);
        return prm.oob_row;
      }
      return static_cast<int>(sl);
    };
    int q = 0;
    bool ok = true;
    // slot kinds: S slot j (0..4) of tile t = features [128 j, +128) of this CTA's keys (j = 4: the rotary 64);
    // V slot v (0..3) of tile t = value features [256 (v >> 1) + 128 r, +128) of keys [128 (v & 1), +128)
    auto issue = [&](int t, bool is_v, int j) {
      const int st = q % NSLOT;
      if (!ok) return;   // after a wait gave up nothing more is issued
      if (q >= NSLOT && !(ok = mbar_wait(bar(B_EMPTY + st), ((q / NSLOT) - 1) & 1, prm.err))) return;
      const uint32_t dst = sb + RING_OFF + st * SLOT;
      const int nblk = (!is_v && j == 4) ? 1 : 2;
      const int key0 = k0 + t * PT + (is_v ? (j & 1) : r) * TK;
      const int f0 = is_v ? ((j >> 1) * 4 + r * 2) : 2 * j;   // first 64-feature block
      const bool sp0 = is_v && holds_last(key0, p), sp1 = is_v && holds_last(key0 + 64, p);
      // both CTAs skip the same groups (the tile and p are common), so CTA 0 can count the pair's bytes
      if (r == 0) mbar_arrive_expect_tx(bar(B_FULL + st), 2 * nblk * (2 - sp0 - sp1) * BOX);
      const int m0 = (is_v ? (j & 1) : r) * 2;   // the slot's first group within the tile
      const int g0 = group_row(t, m0, is_v), g1 = group_row(t, m0 + 1, is_v);
      for (int blk = 0; blk < nblk; ++blk) {
        if (!sp0) tma_load_2d_pair(dst + blk * ATOM, &tmc, full0 + 8u * st, (f0 + blk) * 64, g0);
        if (!sp1) tma_load_2d_pair(dst + blk * ATOM + BOX, &tmc, full0 + 8u * st, (f0 + blk) * 64, g1);
      }
      if (sp0 || sp1) {   // this CTA's copy of the group lands on a local barrier; warp 3 then clears rows past p
        const int fb = j >> 1, hr = sp1 ? 1 : 0;
        fill[fb * 4 + 0] = static_cast<int>(dst + hr * BOX);
        fill[fb * 4 + 1] = key0 + hr * 64;
        mbar_arrive_expect_tx(bar(B_FILL + fb), 2 * BOX);
        const int gr = group_row(t, m0 + hr, false);
        for (int blk = 0; blk < 2; ++blk)
          tma_load_2d(dst + hr * BOX + blk * ATOM, &tmc, bar(B_FILL + fb), (f0 + blk) * 64, gr);
      }
      ++q;
    };
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      lookup(t);
#pragma unroll 1
      for (int j = 0; j < 5; ++j) issue(t, false, j);
      if (t >= 1)
#pragma unroll 1
        for (int v = 0; v < 4; ++v) issue(t - 1, true, v);
    }
#pragma unroll 1
    for (int v = 0; v < 4; ++v) issue(n_tiles - 1, true, v);
    // the pair's MMAs have read every slot this CTA filled (so no copy of it is still in flight)
    for (int i = max(0, q - NSLOT); i < q; ++i) mbar_wait(bar(B_EMPTY + i % NSLOT), (i / NSLOT) & 1, prm.err);
  } else if (warp == 3 && has_split) {
    // ------------------------------------------------------------------ boundary fill (both CTAs)
    // the group's value rows have landed (this CTA's copy, local barrier): zero the rows of keys past p
    const uint32_t split0 = map_to_rank(bar(B_SPLIT), 0);
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
    for (int fb = 0; fb < 2; ++fb) {
      if (!mbar_wait(bar(B_FILL + fb), 0, prm.err)) break;   // the producer gave up before this slot
      const uint32_t dst = static_cast<uint32_t>(fill[fb * 4 + 0]);
      const int first = p - fill[fb * 4 + 1] + 1;   // rows [first, 64) hold keys past p (whole 128-byte rows)
#pragma unroll 1
      for (int e = first * 8 + lane; e < 64 * 8; e += 32) {
        st_shared_v4(dst + e * 16, zero);
        st_shared_v4(dst + ATOM + e * 16, zero);
      }
      fence_proxy_async_smem();   // generic stores before the tensor core reads them
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(split0 + 8u * fb);
    }
  } else if (warp == 1 && lane == 0 && r == 0) {
    // ------------------------------------------------------------------ MMA issuer (CTA 0 for the pair)
    constexpr uint32_t id_s = idesc_bf16_f32(256, 128, false, false);
    constexpr uint32_t id_o = idesc_bf16_f32(256, 128, true, true);
    bool ok = mbar_wait(bar(B_QFULL), 0, prm.err);
    int q = 0;
    auto s_tile = [&](int t) {
      const int b = t & 1;
      if (t >= 2 && ok) ok = mbar_wait_cluster(bar(B_SFREE + b), ((t >> 1) - 1) & 1, prm.err);
      tc_fence_after();
      const uint32_t d = tmem + b * 128;
#pragma unroll 1
      for (int j = 0; j < 5 && ok; ++j) {
        const int st = q % NSLOT;
        ok = mbar_wait(bar(B_FULL + st), (q / NSLOT) & 1, prm.err);
        if (!ok) break;
        tc_fence_after();
        // descriptors advance by the operand's byte offset / 16 (shared memory < 256 KB: no carry out of the
        // address field)
        const uint64_t da = sdesc_sw128(sb + RING_OFF + st * SLOT, 16, 1024);
        const uint64_t db = sdesc_sw128(sb + Q_OFF + 2 * j * BOX, 16, 1024);
        if (j < 4) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss_pair(d, da + (((kk >> 2) * ATOM + (kk & 3) * 32) >> 4), db + (((kk >> 2) * BOX + (kk & 3) * 32) >> 4),
                        id_s, (j | kk) != 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_ss_pair(d, da + ((kk * 32) >> 4), db + ((kk * 32) >> 4), id_s, 1u);
        }
        tc_commit_pair(bar(B_EMPTY + st));
        ++q;
      }
      if (ok) tc_commit_pair(bar(B_SFULL + b));
    };
    auto o_tile = [&](int t) {
      if (ok) ok = mbar_wait_cluster(bar(B_PFULL), t & 1, prm.err);
      tc_fence_after();
#pragma unroll 1
      for (int v = 0; v < 4 && ok; ++v) {
        const int st = q % NSLOT;
        ok = mbar_wait(bar(B_FULL + st), (q / NSLOT) & 1, prm.err);
        if (!ok) break;
        const int key0 = k0 + t * PT + (v & 1) * TK;
        if (holds_last(key0, p) || holds_last(key0 + 64, p)) {   // used once per CTA pair: phase 0
          ok = mbar_wait_cluster(bar(B_SPLIT + (v >> 1)), 0, prm.err);
          if (!ok) break;
        }
        tc_fence_after();
        const uint32_t d = tmem + 256 + (v >> 1) * 128;
        const uint64_t da = sdesc_sw128(sb + RING_OFF + st * SLOT, ATOM, 1024);
        const uint64_t db = sdesc_sw128(sb + PT_OFF + (v & 1) * TK * 128, ATOM, 1024);
        const uint32_t acc0 = (t > 0 || (v & 1)) ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // 16 keys per step: V^T and P^T are MN-major (features, heads contiguous)
          mma_ss_pair(d, da + kk * 128, db + kk * 128, id_o, kk > 0 ? 1u : acc0);
        tc_commit_pair(bar(B_EMPTY + st));
        ++q;
      }
      if (ok) tc_commit_pair(bar(B_ODONE));
    };
#pragma unroll 1
    for (int t = 0; t < n_tiles && ok; ++t) {
      s_tile(t);
      if (t >= 1) o_tile(t - 1);
    }
    if (ok) o_tile(n_tiles - 1);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax and epilogue (both CTAs)
    // eight warps: warp w reads TMEM lane quarter w % 4 (its 32 keys of S^T, its 32 features of O^T) and handles
    // heads [64 hh, +64), hh = (w - 4) / 4; threads 0..127 of the group keep the running max of one head each
    const int q4 = warp & 3;
    const int hh = (warp - 4) >> 2;
    const int kr = q4 * 32 + lane;          // key row of S^T, feature row of O^T
    const int tid = threadIdx.x - 128;
    const bool head_owner = tid < H;
    const int hd = tid & (H - 1);
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t peer = static_cast<uint32_t>(r ^ 1);
    const uint32_t sfree0 = map_to_rank(bar(B_SFREE), 0), pfull0 = map_to_rank(bar(B_PFULL), 0);
    const uint32_t mx_peer = map_to_rank(sb + MX_OFF, peer), mxfull_peer = map_to_rank(bar(B_MXFULL), peer);
    // P^T of heads [64 r, +64) lives in CTA r: this warp's probabilities go to the other CTA when hh != r
    const bool remote = hh != r;
    const uint32_t pt_dst = remote ? map_to_rank(sb + PT_OFF, peer) : sb + PT_OFF;
    float* mx = reinterpret_cast<float*>(smem + MX_OFF);
    float* wm = reinterpret_cast<float*>(smem + WM_OFF);
    float* m_s = reinterpret_cast<float*>(smem + M_OFF);
    float* al_s = reinterpret_cast<float*>(smem + AL_OFF);
    const float zmul = prm.scale * kLog2e;
    float l_acc[2] = {0.f, 0.f};   // this warp's keys, heads 64 hh + 32 jj + lane
    bool ok = true;
#pragma unroll 1
    for (int t = 0; t < n_tiles; ++t) {
      const int b = t & 1;
      const int key = k0 + t * PT + r * TK + kr;
      const bool valid = key >= lo && key < k1;
      if (ok) ok = mbar_wait_cluster(bar(B_SFULL + b), (t >> 1) & 1, prm.err);
      tc_fence_after();
      const uint32_t s_t = tmem + lane_addr + b * 128 + hh * 64;
      // (1) per-head maximum over this CTA's 128 keys, sent to the other CTA (which needs it to decide alike)
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t v[32];
        tmem_ld32(s_t + jj * 32, v);
        tmem_wait_ld();
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = valid ? __uint_as_float(v[e]) : -CUDART_INF_F;
        wm[q4 * H + hh * 64 + jj * 32 + lane] = warp_colreduce32<true>(x, lane);
      }
      bar_sync_softmax();
      float cm = -CUDART_INF_F;
      bool need = false;   // this CTA's keys alone would move the running max
      if (head_owner) {
        cm = fmaxf(fmaxf(wm[hd], wm[H + hd]), fmaxf(wm[2 * H + hd], wm[3 * H + hd]));
        st_cluster_f32(mx_peer + (b * H + hd) * 4, cm);
        __syncwarp();   // the warp's stores precede lane 0's release-arrive
        if (lane == 0) mbar_arrive_cluster(mxfull_peer + 8u * b);
        need = cm != -CUDART_INF_F && cm * zmul > m_reg + kGrow;
      }
      const bool need_any = bar_or_softmax(need);
      // (2) the previous tile's O^T MMAs are done: P^T may be overwritten (and O^T rescaled)
      if (t >= 1 && ok) ok = mbar_wait(bar(B_ODONE), (t - 1) & 1, prm.err);
      tc_fence_after();
      // (3) probabilities of this warp's heads for this CTA's keys (P^T rows r * 128 + key) against the running
      // max, and their sums over the keys; the exchanged maxima are read only after this (their trip between
      // the CTAs overlaps it), and a tile on which the running max moves computes them again
      const int prow = r * TK + kr;
      float lt[2] = {0.f, 0.f};
      auto p_pass = [&]() {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          uint32_t v[32];
          tmem_ld32(s_t + jj * 32, v);
          tmem_wait_ld();
          const float4* m4 = reinterpret_cast<const float4*>(m_s + hh * 64 + jj * 32);
          float x[32];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 m = m4[e4];
            const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              x[4 * e4 + k] = valid ? ex2(fmaf(__uint_as_float(v[4 * e4 + k]), zmul, -mm[k])) : 0.f;
          }
          const uint32_t dst = pt_dst + prow * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 pk;
            pk.x = pack2(x[8 * i + 0], x[8 * i + 1]);
            pk.y = pack2(x[8 * i + 2], x[8 * i + 3]);
            pk.z = pack2(x[8 * i + 4], x[8 * i + 5]);
            pk.w = pack2(x[8 * i + 6], x[8 * i + 7]);
            const uint32_t a = dst + (((jj * 4 + i) ^ (prow & 7)) << 4);
            if (remote)
              st_cluster_v4(a, pk);
            else
              st_shared_v4(a, pk);
          }
          lt[jj] = warp_colreduce32<false>(x, lane);
        }
      };
      if (!need_any) p_pass();   // optimistic: the running max holds unless the other CTA's keys move it
      // (4) the pair's maxima: both CTAs take the same decision per head from the same numbers
      bool grow = false;
      if (head_owner) {
        if (ok) ok = mbar_wait_cluster(bar(B_MXFULL + b), (t >> 1) & 1, prm.err);
        const float gm = fmaxf(cm, mx[b * H + hd]);
        const float gz = gm == -CUDART_INF_F ? -CUDART_INF_F : gm * zmul;
        grow = gz > m_reg + kGrow;
        float alpha = 1.f;
        if (grow) {
          alpha = m_reg == -CUDART_INF_F ? 0.f : ex2(m_reg - gz);
          m_reg = gz;
        }
        m_s[hd] = m_reg == -CUDART_INF_F ? 0.f : m_reg;   // -inf only while every key so far was masked
        al_s[hd] = alpha;
      }
      const bool any_grow = bar_or_softmax(grow);
      if (any_grow) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) l_acc[jj] *= al_s[hh * 64 + jj * 32 + lane];
        if (t >= 1) {
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb) {   // 2 feature blocks x this warp's 2 column groups of 32 heads
            const int h0 = hh * 64 + (cb & 1) * 32;
            const uint32_t o_t = tmem + lane_addr + 256 + (cb >> 1) * 128 + h0;
            uint32_t v[32];
            tmem_ld32(o_t, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * al_s[h0 + e]);
            tmem_st32(o_t, v);
          }
          tmem_wait_st();
        }
        p_pass();   // against the new running max (overwrites the optimistic pass, if any)
      } else if (need_any) {
        p_pass();   // cannot happen (a local need makes the pair's max grow); kept for safety
      }
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) l_acc[jj] += lt[jj];
      tc_fence_before();
      // this thread's P^T stores before the tensor core reads them (the other CTA's memory: cluster scope)
      if (remote)
        fence_proxy_async_cluster();
      else
        fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(sfree0 + 8u * b);   // this S^T buffer may be overwritten
        mbar_arrive_cluster(pfull0);
      }
    }
    // (4) epilogue: unnormalised O (fp32) for this CTA's 256 features and all heads; per-head sums
    if (ok) ok = mbar_wait(bar(B_ODONE), (n_tiles - 1) & 1, prm.err);
    tc_fence_after();
    float* ws = prm.ws_o + (static_cast<long long>(s) * H * prm.n_splits + c) * 512;
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      const int f = (cb >> 1) * 256 + r * 128 + kr;
      const int h0 = hh * 64 + (cb & 1) * 32;
      uint32_t v[32];
      tmem_ld32(tmem + lane_addr + 256 + (cb >> 1) * 128 + h0, v);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        ws[static_cast<long long>(h0 + e) * prm.n_splits * 512 + f] = __uint_as_float(v[e]);
    }
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) wm[q4 * H + hh * 64 + jj * 32 + lane] = l_acc[jj];
    bar_sync_softmax();
    if (head_owner) {
      l_cta = wm[hd] + wm[H + hd] + wm[2 * H + hd] + wm[3 * H + hd];
      if (r == 1) st_cluster_f32(map_to_rank(sb + LP_OFF + hd * 4, 0), l_cta);
    }
  }
  tc_fence_before();
  __syncthreads();
  // every MMA, copy, commit and remote store of the pair has landed before either CTA passes this point
  cluster_sync();
  tc_fence_after();
  if (r == 0 && warp >= 4 && warp < 8) {
    const int hd = threadIdx.x - 128;
    const float l_peer = reinterpret_cast<const float*>(smem + LP_OFF)[hd];
    prm.ws_ml[(static_cast<long long>(s) * H + hd) * prm.n_splits + c] = make_float2(m_reg, l_cta + l_peer);
  }
  if (warp == 2) tmem_dealloc_pair(tmem, 512);
}

}  // namespace mlap

int mla_pair_chunk(int n_seqs, int max_keys) {
#ifdef DA_TUNING_HOOKS
  const char* env = std::getenv("DA_MLA_CHUNK");   // sweep override in tuning builds only (multiple of 256)
  if (env && std::atoi(env) >= mlap::PT && std::atoi(env) % mlap::PT == 0) return std::atoi(env);
#endif
  int chunk = mlap::PT;
  // grow the chunk (fewer partials) while the grid keeps >= 4 waves of the 76 CTA pairs a 152-SM part holds
  while (chunk < 16384 && static_cast<long long>(n_seqs) * ((max_keys + 2 * chunk - 1) / (2 * chunk)) >= 4LL * 76)
    chunk *= 2;
  return chunk;
}

cudaError_t launch_mla_pair_decode(const MlaArgs& a, const MlaPlan& plan, float* ws_o, float2* ws_ml,
                                   cudaStream_t stream) {
  using namespace mlap;
  if (a.hq != H || plan.chunk % PT != 0) return cudaErrorInvalidValue;
  CUtensorMap tmq, tmc;
  const uint64_t rows_total = a.block_table ? static_cast<uint64_t>(a.n_blocks) * a.block_size
                                            : static_cast<uint64_t>(a.num_rows) * a.max_len;
  if (rows_total + 512 > 0x7fffffffULL) return cudaErrorInvalidValue;   // TMA row coordinates are int32
  if (!encode_tmap_2d_bf16(&tmq, a.q, DR, static_cast<uint64_t>(a.n_seqs) * H, DR * 2, 64, HH) ||
      !encode_tmap_2d_bf16(&tmc, a.cache, DR, rows_total, DR * 2, 64, 64))
    return cudaErrorInvalidValue;
  Params prm;
  prm.rows = a.rows;
  prm.positions = a.positions;
  prm.ws_o = ws_o;
  prm.ws_ml = ws_ml;
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
  prm.oob_row = static_cast<int>(rows_total);
  prm.err = a.err;
  // per device and cheap: set on every launch
  cudaError_t ea = cudaFuncSetAttribute(mla_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (ea != cudaSuccess) return ea;
  return launch_dependent(mla_pair_kernel, dim3(2 * plan.n_splits, 1, a.n_seqs), dim3(THREADS), SMEM_BYTES, stream, tmq,
                          tmc, prm);
}

}  // namespace da
