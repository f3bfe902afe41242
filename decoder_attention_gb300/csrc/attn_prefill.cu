// Prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16 operands, fp32 softmax.
//
// Computes causal_attention of DecoderAttention.forward for prefill chunks (page "42. More models: a
// registry, scaled RoPE, sliding windows and latent attention", sections "What differs between model
// families" and "Sliding windows"; soft-capping as "Model resolution" lists it for Gemma 2): for every
// query row, softmax over its visible keys of scale * q.k (optionally c * tanh(. / c)), times V.
//
// CTA = 256 query rows (two 128-row tiles Q0, Q1) of one (sequence, query head). Key tiles of 128 keys
// stream by TMA (128-byte swizzle) through a 2-stage ring whose stage holds one round's K and V tiles.
// Roles:
//   warp 8      TMA producer of Q (once) and K tiles
//   warp 10     TMA producer of V tiles
//   warp 9      MMA issuer (one thread): S_w = Q_w K^T into TMEM; O_w += P_w V with P_w read from TMEM
//   warp 11     idle (completes the third warpgroup, which setmaxnreg works on)
//   warps 0-3   softmax of Q0 rows, warps 4-7 softmax of Q1 rows: one thread per row; S row from TMEM,
//               mask only on tiles that need it, online softmax in fp32 (log2 domain; O is rescaled only
//               when the running max grows by more than 2^8), P written back into TMEM as bf16
// MMA order per key tile j:  PV0(j), S0(j+1), PV1(j), S1(j+1)  -- so the softmax of one Q tile runs while
// the tensor core works on the other tile's PV and next S. S0(j+1) overwrites the TMEM columns of P0(j);
// tcgen05.mma instructions of one thread execute in issue order, so PV0(j) has read P0(j) by then.
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
constexpr int NS = 2;               // ring stages; stage of round slot j holds K(tbeg + j) and V(tbeg + j - 1)
constexpr int THREADS = 384;        // 3 warpgroups: softmax Q0, softmax Q1, producers/MMA
// setmaxnreg split: launched at 168 per thread (384 x 168 = 64512); softmax warpgroups rise to 216 and
// the producer/MMA warpgroup drops to 72: 256 x 216 + 128 x 72 = 64512, the launch total (per SMSP, one
// warp of each warpgroup: 216 + 216 + 72 = 504 of 512 registers per lane).
#ifndef DA_PF_REGS_SOFTMAX
#define DA_PF_REGS_SOFTMAX 216
#define DA_PF_REGS_CTRL 72
#endif
constexpr int REGS_SOFTMAX = DA_PF_REGS_SOFTMAX;
constexpr int REGS_CTRL = DA_PF_REGS_CTRL;
static_assert(256 * REGS_SOFTMAX + 128 * REGS_CTRL == 384 * 168, "register split must match the launch total");
constexpr int HALF = 128 * 128;     // bytes of a 64-wide half of a 128-row tile (16 KB)
constexpr int TILE = 2 * HALF;      // 32 KB
constexpr int OFF_Q = 0;
constexpr int OFF_R = OFF_Q + NQT * TILE;   // ring: stage s = K tile at OFF_R + 2s TILE, V tile after it
constexpr int OFF_BAR = OFF_R + NS * 2 * TILE;
// barriers: q[NQT], full[NS] (two arrivals: K producer, V producer), empty[NS], s_full[NQT], p_full[NQT],
// o_done[NQT]
constexpr int B_Q = 0, B_FU = B_Q + NQT, B_EM = B_FU + NS, B_SF = B_EM + NS,
              B_PF = B_SF + NQT, B_OD = B_PF + NQT, N_BARS = B_OD + NQT;
constexpr int SMEM_BYTES = OFF_BAR + N_BARS * 8 + 16 + 1024;   // + TMEM address slot + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
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

// 32 lanes x 128 consecutive 32-bit columns in one tcgen05.ld (one tensor-memory request per warp instead
// of four; the MMA issuer's tcgen05 operations queue behind the softmax warps' loads and stores).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127"
      "}, [%128];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr));
}

// 32 lanes x 64 consecutive 32-bit columns in one tcgen05.st.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64"
      "};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63]) : "memory");
}

// One pass over a row's 128 scores: soft-cap (CAP), mask to the visible column range [lo_c, hi_c] (MASK),
// and the row max with 8 independent partial maxima (one running max would be a 128-long dependency chain).
template <bool CAP, bool MASK>
__device__ __forceinline__ float row_pass(uint32_t (&zr)[BN], float cap_in, float cap_l2, int lo_c, int hi_c) {
  if (CAP || MASK) {
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      float v = __uint_as_float(zr[c]);
      if (CAP) v = cap_l2 * tanh_fast(v * cap_in);
      if (MASK) v = (c >= lo_c && c <= hi_c) ? v : -CUDART_INF_F;
      zr[c] = __float_as_uint(v);
    }
  }
  // 8 independent partial maxima, two new scores per 3-input max
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = fmaxf(__uint_as_float(zr[2 * e]), __uint_as_float(zr[2 * e + 1]));
#pragma unroll
  for (int c = 16; c < BN; c += 2)
    mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], __uint_as_float(zr[c]), __uint_as_float(zr[c + 1]));
  return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

// The 8 MMAs (K = 16 each) of S = Q K^T for one 128 x 128 tile; both operands K-major, 128-byte swizzled
// in two 64-wide halves. One asm block with the descriptors stepped by immediate adds: the issuing thread
// shares its SM sub-partition with two softmax warps, and every instruction between MMAs delays the next.
// The start-address field of a descriptor holds address >> 4 in bits [0, 14); shared addresses stay below
// 2^18, so adding to the low word never carries out of the field. Steps per K = 16 slice (16-byte units):
// 32 bytes within a 128-byte row, then the second 64-wide half 16 KB on.
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, false);
  const uint64_t a = sdesc_sw128(q_smem, 16, 1024), b = sdesc_sw128(k_smem, 16, 1024);
  asm volatile(
      "{\n\t"
      ".reg .b32 alo, ahi, blo, bhi, x, y;\n\t"
      ".reg .b64 da, db;\n\t"
      ".reg .pred pf, pt;\n\t"
      "setp.ne.b32 pf, %3, %3;\n\t"
      "setp.eq.b32 pt, %3, %3;\n\t"
      "mov.b64 {alo, ahi}, %1;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pf;\n\t"
#define DA_S_STEP(o)                                                        \
      "add.u32 x, alo, " #o "; add.u32 y, blo, " #o ";\n\t"                 \
      "mov.b64 da, {x, ahi}; mov.b64 db, {y, bhi};\n\t"                     \
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, pt;\n\t"
      DA_S_STEP(2) DA_S_STEP(4) DA_S_STEP(6) DA_S_STEP(1024) DA_S_STEP(1026) DA_S_STEP(1028) DA_S_STEP(1030)
#undef DA_S_STEP
      "}" ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc)
      : "memory");
}

// The 8 MMAs (K = 16 keys each) of O (+)= P V; P from TMEM (bf16, 2 per column: 8 columns per slice), V
// MN-major in smem (16 key rows = 2048 bytes per slice). One asm block, as for issue_s.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(BM, D, false, true);
  const uint64_t b = sdesc_sw128(v_smem, HALF, 1024);
  asm volatile(
      "{\n\t"
      ".reg .b32 blo, bhi, x, y;\n\t"
      ".reg .b64 db;\n\t"
      ".reg .pred p0, pt;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\t"
      "setp.eq.b32 pt, %3, %3;\n\t"
      "mov.b64 {blo, bhi}, %2;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
#define DA_PV_STEP(ta, o)                                                   \
      "add.u32 x, %1, " #ta "; add.u32 y, blo, " #o ";\n\t"                 \
      "mov.b64 db, {y, bhi};\n\t"                                           \
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [x], db, %3, pt;\n\t"
      DA_PV_STEP(8, 128) DA_PV_STEP(16, 256) DA_PV_STEP(24, 384) DA_PV_STEP(32, 512) DA_PV_STEP(40, 640)
      DA_PV_STEP(48, 768) DA_PV_STEP(56, 896)
#undef DA_PV_STEP
      "}" ::"r"(o_tmem), "r"(p_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmq,
                                                             const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const __grid_constant__ CUtensorMap tmo,
                                                             const Params prm) {
  extern __shared__ uint8_t smem_raw[];
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

  // Key-tile range of each Q tile: from the tile holding the oldest query's first visible key to the tile
  // holding the newest query's own key. Q0's range starts no later and ends no later than Q1's.
  bool valid0, valid1;
  int pmin0, pmax0, pmin1, pmax1, tb0, te0, tb1, te1;
  {
    auto range = [&](int w, bool& valid, int& pmin, int& pmax, int& tb, int& te) {
      const int r0 = q0 + w * BM;
      valid = r0 < n_b;
      const int nr = valid ? min(BM, n_b - r0) : 1;
      pmin = fp + r0;
      pmax = fp + r0 + nr - 1;
      const int lo = window > 0 ? max(0, pmin - window + 1) : 0;
      tb = lo / BN;
      te = pmax / BN;
    };
    range(0, valid0, pmin0, pmax0, tb0, te0);
    range(1, valid1, pmin1, pmax1, tb1, te1);
  }
  const int tbeg = tb0;
  const int tend = valid1 ? te1 : te0;
  const int n_tiles = tend - tbeg + 1;
  auto act0 = [&](int t) { return t >= tb0 && t <= te0; };
  auto act1 = [&](int t) { return valid1 && t >= tb1 && t <= te1; };

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + OFF_BAR;
  auto B = [&](int i) { return bar + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + N_BARS * 8);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(B(B_FU + i), 2);
      mbar_init(B(B_EM + i), 1);
    }
    for (int w = 0; w < NQT; ++w) {
      mbar_init(B(B_SF + w), 1);
      mbar_init(B(B_PF + w), BM);
      mbar_init(B(B_OD + w), 1);
      mbar_init(B(B_Q + w), 1);
    }
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
  const int plane = (row * prm.hkv + g) * prm.max_len;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer: Q and K tiles
      // Round slot j (one ring stage) holds K(tbeg + j) and V(tbeg + j - 1): the K tile the round's scores
      // need and the V tile its PVs need. This producer fills the K halves (slot n_tiles has none: a bare
      // arrival). Q0 and the first K tile go first; Q1 queues behind them.
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      auto load_q = [&](int w) {
        const int tok = t0 + q0 + w * BM;
        mbar_arrive_expect_tx(B(B_Q + w), TILE);
        tma_load_3d(sbase + OFF_Q + w * TILE, &tmq, B(B_Q + w), 0, h, tok);
        tma_load_3d(sbase + OFF_Q + w * TILE + HALF, &tmq, B(B_Q + w), 64, h, tok);
      };
      load_q(0);
      bool q1_loaded = false;
      int issued = 0;
      for (int j = 0; j <= n_tiles && !*vabort; ++j) {
        if (j == 1 && valid1) {
          load_q(1);
          q1_loaded = true;
        }
        const int st = j % NS;
        if (j >= NS && !mbar_wait(B(B_EM + st), ((j / NS) + 1) & 1, prm.err)) {
          abort_flag = 1;
          break;
        }
        if (j < n_tiles) {
          const int key = plane + (tbeg + j) * BN;
          const uint32_t dst = sbase + OFF_R + st * 2 * TILE;
          mbar_arrive_expect_tx(B(B_FU + st), TILE);
          tma_load_2d(dst, &tmk, B(B_FU + st), 0, key);
          tma_load_2d(dst + HALF, &tmk, B(B_FU + st), 64, key);
        } else {
          mbar_arrive(B(B_FU + st));
        }
        ++issued;
      }
      if (valid1 && !q1_loaded && !*vabort) {
        load_q(1);
        q1_loaded = true;
      }
      // every issued copy must land before the CTA's shared memory is released
      mbar_wait(B(B_Q + 0), 0, prm.err);
      if (q1_loaded) mbar_wait(B(B_Q + 1), 0, prm.err);
      for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(B(B_FU + j % NS), (j / NS) & 1, prm.err);
    } else if (warp == 10 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer: V tiles
      // the V halves of the round slots (slot 0 has none: a bare arrival)
      prefetch_tmap(&tmv);
      int issued = 0;
      for (int j = 0; j <= n_tiles && !*vabort; ++j) {
        const int st = j % NS;
        if (j >= NS && !mbar_wait(B(B_EM + st), ((j / NS) + 1) & 1, prm.err)) {
          abort_flag = 1;
          break;
        }
        if (j > 0) {
          const int key = plane + (tbeg + j - 1) * BN;
          const uint32_t dst = sbase + OFF_R + st * 2 * TILE + TILE;
          mbar_arrive_expect_tx(B(B_FU + st), TILE);
          tma_load_2d(dst, &tmv, B(B_FU + st), 0, key);
          tma_load_2d(dst + HALF, &tmv, B(B_FU + st), 64, key);
        } else {
          mbar_arrive(B(B_FU + st));
        }
        ++issued;
      }
      for (int j = max(0, issued - NS); j < issued; ++j) mbar_wait(B(B_FU + j % NS), (j / NS) & 1, prm.err);
    } else if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer (one thread)
      const uint32_t q0s = sbase + OFF_Q, q1s = sbase + OFF_Q + TILE;
      const uint32_t s0t = tmem, s1t = tmem + BN, o0t = tmem + 256, o1t = tmem + 256 + D;
      int npv0 = 0, npv1 = 0;
      bool od0 = false;
      bool q1_ready = false;
      auto wait_q1 = [&]() {          // Q1 lands after the first K tile; waited on before its first scores
        if (!q1_ready) {
          q1_ready = mbar_wait(B(B_Q + 1), 0, prm.err);
          tc_fence_after();
        }
        return q1_ready;
      };
      bool ok = mbar_wait(B(B_Q + 0), 0, prm.err) && mbar_wait(B(B_FU), 0, prm.err);
      tc_fence_after();
      if (ok) {
        // prologue: scores of the first key tile
        if (act0(tbeg)) {
          issue_s(s0t, q0s, sbase + OFF_R);
          tc_commit(B(B_SF + 0));
        }
        if (act1(tbeg)) {
          ok = wait_q1();
          if (ok) {
            issue_s(s1t, q1s, sbase + OFF_R);
            tc_commit(B(B_SF + 1));
          }
        }
        tc_commit(B(B_EM + 0));
      }
      // Per round (key tile t): PV0(t), S0(t+1), PV1(t), S1(t+1), all reading round slot i + 1 (V(t) and
      // K(t+1)), which one commit releases at the end. Each tcgen05.mma blocks the issuing thread until the
      // tensor core takes it (the queue is short), so any wait between two MMA groups idles the tensor
      // core: the operand waits (the slot, Q1), normally satisfied long before, sit at the top of the
      // round while the previous round's last group still runs, and between groups there are only the P
      // waits. The slot's stage and phase advance by counting, not dividing.
      int st = 1 % NS, ph = (1 / NS) & 1;
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int t = tbeg + i;
        const bool nxt = i + 1 < n_tiles;
        const uint32_t k1s = sbase + OFF_R + st * 2 * TILE;
        const uint32_t vs = k1s + TILE;
        if (!mbar_wait(B(B_FU + st), ph, prm.err) || (nxt && act1(t + 1) && !wait_q1())) {
          ok = false;
          break;
        }
        if (act0(t)) {
          if (!mbar_wait(B(B_PF + 0), npv0 & 1, prm.err)) { ok = false; break; }
          tc_fence_after();
          issue_pv(o0t, s0t, vs, npv0 > 0);
          ++npv0;
          if (t == te0) {
            tc_commit(B(B_OD + 0));     // Q0's output is final: its epilogue overlaps Q1's last tiles
            od0 = true;
          }
        }
        if (nxt && act0(t + 1)) {
          issue_s(s0t, q0s, k1s);
          tc_commit(B(B_SF + 0));
        }
        if (act1(t)) {
          if (!mbar_wait(B(B_PF + 1), npv1 & 1, prm.err)) { ok = false; break; }
          tc_fence_after();
          issue_pv(o1t, s1t, vs, npv1 > 0);
          ++npv1;
        }
        if (nxt && act1(t + 1)) {
          issue_s(s1t, q1s, k1s);
          tc_commit(B(B_SF + 1));
        }
        tc_commit(B(B_EM + st));
        if (++st == NS) {
          st = 0;
          ph ^= 1;
        }
      }
      if (!ok) abort_flag = 1;
      if (!od0) tc_commit(B(B_OD + 0));
      tc_commit(B(B_OD + 1));
      mbar_wait(B(B_OD + 1), 0, prm.err);   // all MMAs done before TMEM may be released
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
    const float cap_in = cap > 0.f ? prm.scale / cap : 0.f;
    const float cap_l2 = cap * kLog2e;
    const float zmul = cap > 0.f ? 1.f : prm.scale * kLog2e;   // z * zmul is the logit in log2 units
    const bool my_valid = w == 0 ? true : valid1;
    const int my_tb = w == 0 ? tb0 : tb1;
    const int my_te = w == 0 ? te0 : te1;
    const int my_pmin = w == 0 ? pmin0 : pmin1;
    const int my_pmax = w == 0 ? pmax0 : pmax1;
    float m = -CUDART_INF_F, l = 0.f;
    int nact = 0;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int t = tbeg + i;
      if (!my_valid || t < my_tb || t > my_te) continue;
      // outcomes are made warp-uniform: the TMEM loads and stores below are warp-collective
      if (__any_sync(0xffffffffu, *vabort != 0)) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(B(B_SF + w), nact & 1, prm.err))) {
        abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t zr[BN];
#pragma unroll
      tmem_ld128(t_s, zr);
      tmem_wait_ld();
      const int kstart = t * BN;
      const bool need_mask = !(kstart + BN - 1 <= my_pmin &&
                               (window == 0 || my_pmax - kstart <= window - 1) && kstart + BN <= kv_len);
      // zr: the raw score q.k (scaled into log2 units inside the exponent), or for capped layers the
      // capped logit already in log2 units. Visible keys of this row in the tile: columns [lo_c, hi_c].
      const int hi_c = min(p, kv_len - 1) - kstart;
      const int lo_c = window > 0 ? p - window + 1 - kstart : -BN;
      float tmax;
      if (cap > 0.f) {
        tmax = need_mask ? row_pass<true, true>(zr, cap_in, cap_l2, lo_c, hi_c)
                         : row_pass<true, false>(zr, cap_in, cap_l2, lo_c, hi_c);
      } else {
        tmax = need_mask ? row_pass<false, true>(zr, cap_in, cap_l2, lo_c, hi_c)
                         : row_pass<false, false>(zr, cap_in, cap_l2, lo_c, hi_c);
      }
      tmax *= zmul;
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
      const float nmu = (m == -CUDART_INF_F) ? 0.f : -m;
      // p = 2^(z * zmul - m) two scores at a time (packed fp32 pairs), row sum in 4 packed accumulators
      const uint64_t zmul2 = f2_pack(zmul, zmul), nmu2 = f2_pack(nmu, nmu);
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[BN / 2];
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        float xa, xb;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(zr[2 * e]), __uint_as_float(zr[2 * e + 1])), zmul2, nmu2), xa, xb);
        const float pa = ex2(xa), pb = ex2(xb);
        ls2[e & 3] = f2_add(ls2[e & 3], f2_pack(pa, pb));
        pk[e] = pack_bf16(pa, pb);
      }
      tmem_st64(t_s, pk);     // P (bf16, 2 per column) over the first half of the S columns
      {
        float a0, a1, b0, b1, c0, c1, d0, d1;
        f2_unpack(f2_add(ls2[0], ls2[1]), a0, a1);
        f2_unpack(f2_add(ls2[2], ls2[3]), b0, b1);
        (void)c0; (void)c1; (void)d0; (void)d1;
        l += (a0 + a1) + (b0 + b1);
      }
      tmem_wait_st();
      if (kstart + BN > kv_len) {
        // V rows past the row's last key hold whatever the cache holds there (maybe NaN); P is 0 there,
        // but 0 * NaN is NaN, so zero those rows before the tensor core reads them (after the V copy has
        // landed; the stage cannot be refilled before this tile's PV, which waits for us).
        if (!__all_sync(0xffffffffu, mbar_wait(B(B_FU + (i + 1) % NS), ((i + 1) / NS) & 1, prm.err))) {
          abort_flag = 1;
          ok = false;
          break;
        }
        if (kstart + r >= kv_len) {
          uint8_t* vtile = smem + OFF_R + ((i + 1) % NS) * 2 * TILE + TILE;   // V(t), in round slot i + 1
          uint4* vrow0 = reinterpret_cast<uint4*>(vtile + r * 128);
          uint4* vrow1 = reinterpret_cast<uint4*>(vtile + HALF + r * 128);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            vrow0[e] = make_uint4(0, 0, 0, 0);
            vrow1[e] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(B(B_PF + w));
      ++nact;
    }
    // ------------------------------------------------------------ epilogue: O / l -> out
    // Each warp normalises its 32 rows into the Q tile's shared memory (free once every MMA is done) in the
    // 128-byte-swizzled layout and writes them with two TMA tensor stores; a warp whose rows run past the
    // chunk stores row by row instead (a whole box would overwrite the next sequence's rows).
    if (ok && __all_sync(0xffffffffu, mbar_wait(B(B_OD + w), 0, prm.err))) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool full_tile = q0 + w * BM + wi * 32 + 32 <= n_b;   // warp-uniform
      uint4* orow = reinterpret_cast<uint4*>(prm.out + (static_cast<long long>(t0 + qrow) * prm.hq + h) * D);
      uint8_t* srow = smem + OFF_Q + w * TILE + r * 128;
#pragma unroll
      for (int j = 0; j < D / 32; ++j) {
        uint32_t ov[32];
        tmem_ld32(t_o + j * 32, ov);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint4 u;
          u.x = pack_bf16(__uint_as_float(ov[8 * e + 0]) * inv_l, __uint_as_float(ov[8 * e + 1]) * inv_l);
          u.y = pack_bf16(__uint_as_float(ov[8 * e + 2]) * inv_l, __uint_as_float(ov[8 * e + 3]) * inv_l);
          u.z = pack_bf16(__uint_as_float(ov[8 * e + 4]) * inv_l, __uint_as_float(ov[8 * e + 5]) * inv_l);
          u.w = pack_bf16(__uint_as_float(ov[8 * e + 6]) * inv_l, __uint_as_float(ov[8 * e + 7]) * inv_l);
          const int c16 = j * 4 + e;                 // 16-byte chunk of the row, 0..15
          if (full_tile) {
            *reinterpret_cast<uint4*>(srow + (c16 >> 3) * HALF + (((c16 & 7) ^ (r & 7)) << 4)) = u;
          } else if (row_ok) {
            orow[c16] = u;
          }
        }
      }
      if (full_tile) {
        fence_proxy_async_smem();                    // generic-proxy writes -> visible to the copy engine
        __syncwarp();
        if (lane == 0) {
          const uint32_t src = sbase + OFF_Q + w * TILE + wi * 32 * 128;   // 4 KB aligned: swizzle phase 0
          const int tok = t0 + q0 + w * BM + wi * 32;
          tma_store_3d(&tmo, src, 0, h, tok);
          tma_store_3d(&tmo, src + HALF, 64, h, tok);
          bulk_commit();
          bulk_wait_read();                          // shared memory stays valid until the copies read it
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
  CUtensorMap tmq, tmk, tmv, tmo;
  const uint64_t rows_total = static_cast<uint64_t>(a.num_rows) * a.hkv * a.max_len;
  // q_rot and out [N, Hq, D]: q rows past N are zero-filled by the copy engine, never read from memory; out
  // boxes are only stored whole when all their rows belong to the chunk
  const uint64_t n_tok = static_cast<uint64_t>(a.n_tokens);
  if (!encode_tmap_3d_bf16(&tmq, a.q_rot, D, a.hq, n_tok, D * 2, static_cast<uint64_t>(a.hq) * D * 2, 64, 1, BM) ||
      !encode_tmap_3d_bf16(&tmo, a.out, D, a.hq, n_tok, D * 2, static_cast<uint64_t>(a.hq) * D * 2, 64, 1, 32) ||
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
  prefill_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(tmq, tmk, tmv, tmo, prm);
  return cudaGetLastError();
}

}  // namespace da
