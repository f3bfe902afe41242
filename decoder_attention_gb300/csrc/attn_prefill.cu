// Prefill attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA), bf16 operands, fp32 softmax.
//
// Computes causal_attention of DecoderAttention.forward for prefill chunks (page "42. More models: a
// registry, scaled RoPE, sliding windows and latent attention", sections "What differs between model
// families" and "Sliding windows"; soft-capping as "Model resolution" lists it for Gemma 2): for every
// query row, softmax over its visible keys of scale * q.k (optionally c * tanh(. / c)), times V.
//
// Persistent: one CTA per SM walks a fixed list of work items. An item is two 128-row query tiles Q0, Q1
// that read the same KV head: the same 128 rows of two query heads when the heads per KV head are even
// (both tiles then see the same key tiles), else 256 consecutive rows of one head. Every CTA ranks the
// items by key-tile count and takes its share in snake order. The items' key tiles form one sequence that
// streams by TMA (128-byte swizzle) through a 2-stage ring; a stage holds one round's K and V tiles. Each Q
// tile's buffer is freed as soon as its last scores are done, so the next item's Q tiles load while the
// current item finishes; the output leaves through a per-warp staging slot by TMA tensor stores. Roles:
//   warp 11     item decoder: reads the chunk tables into a small ring of decoded items in shared memory
//               that every other role walks in the same order
//   warp 8      TMA producer of Q tiles and of the K halves of the ring
//   warp 10     TMA producer of the V halves of the ring
//   warp 9      MMA issuer (one thread): S_w = Q_w K^T into TMEM; O_w += P_w V with P_w read from TMEM
//   warps 0-3   softmax of Q0 rows, warps 4-7 softmax of Q1 rows: one thread per row; S row from TMEM,
//               mask only on tiles that need it, online softmax in fp32 (log2 domain; O is rescaled only
//               when the running max grows by more than 2^8), P written back into TMEM as bf16. An item's
//               output O / l leaves during the warpgroup's next item (read from TMEM before its first P
//               arrival), through the warp's staging slot, so that it is off the MMA chain's critical path
// MMA order per round (key tile t, next tile u -- the first tile of the next item after an item's last):
//   PV0(t), S0(u), PV1(t), S1(u)
// so the softmax of one Q tile runs while the tensor core works on the other tile's PV and next S, and at
// an item boundary the next item's scores start while the current item's last softmax runs. S_w(u)
// overwrites the TMEM columns of P_w(t); tcgen05.mma instructions of one thread execute in issue order, so
// PV_w(t) has read P_w(t) by then. TMEM columns: S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512). Key
// tiles outside every query's causal window are never loaded, so a windowed layer costs O(w) per query.
// Every wait is bounded; a wait that gives up sets the device error word and the CTA drains and exits.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {
namespace pf {

constexpr int BM = 128;             // rows per Q tile
constexpr int BN = 128;             // keys per K/V tile
constexpr int D = 128;
constexpr int NQT = 2;              // Q tiles per item
constexpr int NQB = 2;              // Q buffers (each freed by its last scores)
constexpr int NS = 2;               // ring stages
constexpr int NI = 8;               // decoded-item ring entries
constexpr int THREADS = 384;        // 3 warpgroups: softmax Q0, softmax Q1, decoder/producers/MMA
// setmaxnreg split: launched at 168 per thread (384 x 168 = 64512); softmax warpgroups rise to 216 and
// the control warpgroup drops to 72: 256 x 216 + 128 x 72 = 64512, the launch total (per SMSP, one
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
constexpr int OFF_R = OFF_Q + NQB * TILE;   // ring: stage s = K tile at OFF_R + 2s TILE, V tile after it
constexpr int OFF_E = OFF_R + NS * 2 * TILE;  // output staging: 4 KB (16 rows) per softmax warp
constexpr int STG = 16 * 2 * 128;
constexpr int OFF_BAR = OFF_E + 8 * STG;
// barriers: q_full[NQB], q_empty[NQB], full[NS] (two arrivals: K producer, V producer), empty[NS],
// s_full[NQT], p_full[NQT], o_done[NQT], item_full[NI], item_empty[NI], drain
constexpr int B_QF = 0, B_QE = B_QF + NQB, B_FU = B_QE + NQB, B_EM = B_FU + NS, B_SF = B_EM + NS,
              B_PF = B_SF + NQT, B_OD = B_PF + NQT, B_IF = B_OD + NQT, B_IE = B_IF + NI, B_DR = B_IE + NI,
              N_BARS = B_DR + 1;
constexpr int OFF_ITEMS = (OFF_BAR + N_BARS * 8 + 15) / 16 * 16;
constexpr int OFF_SLOT = OFF_ITEMS + NI * 32;
constexpr int kMaxPairs = 512;                     // (chunk, q-tile) pairs the schedule table ranks
constexpr int OFF_ORD = OFF_SLOT + 16;             // schedule table: pair of each cost rank (uint16)
constexpr int SMEM_BYTES = OFF_ORD + kMaxPairs * 2 + 1024;   // + alignment slack
// scratch of the schedule build, in the output staging area: pair costs, then one counter per cost
constexpr int kMaxCostBins = (8 * STG - kMaxPairs * 4) / 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
constexpr uint32_t TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: stale max allowed to lag by up to x256
// readers of every item-ring entry: the two producers, the MMA issuer, the 256 softmax threads
constexpr int kItemReaders = 3 + 256;

struct Params {
  const int32_t* q_start;
  const int32_t* rows;
  const int32_t* first_pos;
  __nv_bfloat16* out;
  int hq, hkv, max_len, num_rows, window;
  int n_seqs, n_qt, n_items;
  int hpair;   // 1: an item is 128 rows of two query heads sharing a KV head; 0: 256 rows of one head
  float softcap, scale;
  const float* sinks;   // [Hq] sink logits (natural units) or NULL
  const int32_t* block_table;   // paged pool: [num_rows, max_blocks] block ids; NULL: contiguous cache
  int block_size, max_blocks, n_blocks;
  int kbox;             // key rows per K/V box: BN, or 64 for pools whose blocks are not multiples of BN
  int* err;
};

// A decoded work item as the ring holds it.
struct Item {
  int t0;      // first token of the chunk
  int n_b;     // chunk length
  int q0;      // first chunk row of the item
  int fp;      // position of the chunk's first token
  int plane;   // contiguous cache: row index of (row, kv head, position 0); paged pool: row * Hkv + kv head
  int h;       // query head
  int kind;    // kEnd, kLive, kBad
  int round0;  // global round of the item's first key tile (rounds count the CTA's key tiles in order)
};
constexpr int kEnd = 0, kLive = 1, kBad = 2;

// The two Q tiles of an item. Head-pair items (query heads per KV head even): the same 128 chunk rows of
// query heads h and h + 1, which share a KV head, so both tiles see the same key tiles. Row-pair items: chunk
// rows q0 .. q0 + 255 of head h, Q1 the upper 128 (its causal range one key tile longer).
__device__ __forceinline__ int qt_row(const Item& it, int w, int hpair) { return it.q0 + (hpair ? 0 : w * BM); }
__device__ __forceinline__ int qt_head(const Item& it, int w, int hpair) { return it.h + (hpair ? w : 0); }

// Key-tile ranges of an item's two Q tiles: each from the tile holding its oldest query's first visible
// key to the tile holding its newest query's own key. Q0's range starts and ends no later than Q1's, and
// together they cover tb0 .. max(te0, te1) without a gap.
struct Tiles {
  bool valid1;             // Q1 has rows
  int pmin0, pmax0, pmin1, pmax1;
  int tb0, te0, tb1, te1;  // tile ranges (te1 < tb1 when Q1 has no rows)
  int n;                   // tiles tb0 .. max(te0, te1)
};
__device__ __forceinline__ Tiles tiles_of(const Item& it, int window, int hpair) {
  Tiles T;
  T.valid1 = hpair || it.q0 + BM < it.n_b;
  const int nr0 = min(BM, it.n_b - it.q0);
  T.pmin0 = it.fp + it.q0;
  T.pmax0 = T.pmin0 + nr0 - 1;
  T.pmin1 = hpair ? T.pmin0 : T.pmin0 + BM;
  T.pmax1 = hpair ? T.pmax0 : T.valid1 ? it.fp + min(it.q0 + 2 * BM, it.n_b) - 1 : T.pmin1;
  T.tb0 = (window > 0 ? max(0, T.pmin0 - window + 1) : 0) / BN;
  T.te0 = T.pmax0 / BN;
  T.tb1 = (window > 0 ? max(0, T.pmin1 - window + 1) : 0) / BN;
  T.te1 = T.valid1 ? T.pmax1 / BN : T.tb1 - 1;
  T.n = (T.valid1 ? T.te1 : T.te0) - T.tb0 + 1;
  return T;
}

// Schedule rank of the item CTA c of G takes in its round r: a snake over the ranks, so that CTAs that take
// a heavier item in one round take a lighter one in the next.
__device__ __forceinline__ int item_of(int r, int c, int G) { return r * G + ((r & 1) ? G - 1 - c : c); }

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

// Soft-cap of a row's 128 raw scores: zr <- tanh(z * cap_in), cap_in = scale / cap, so that cap_l2 * zr is
// the capped logit cap * tanh(scale z / cap) in log2 units; the softmax folds the factor cap_l2 into its
// exponent's FMA (and into the row max, cap_l2 > 0). One packed multiply per two scores and one MUFU tanh
// per score: the soft-capped layer's softmax is bound by the MUFU pipe and the softmax warps' issue.
__device__ __forceinline__ void cap_pass(uint32_t (&zr)[BN], float cap_in) {
  const uint64_t k2 = f2_pack(cap_in, cap_in);
#pragma unroll
  for (int c = 0; c < BN; c += 2) {
    float a, b;
    f2_unpack(f2_mul(f2_pack(__uint_as_float(zr[c]), __uint_as_float(zr[c + 1])), k2), a, b);
    zr[c] = __float_as_uint(tanh_approx(a));
    zr[c + 1] = __float_as_uint(tanh_approx(b));
  }
}

// Soft-cap on the FMA pipe for tiles whose scores are all small: tanh(u) = u * P(u^2) with a cubic P fitted
// here to minimise the relative error over |u| <= kCapPolyRange (6.2e-7 evaluated in fp32, against 1e-5 for the
// MUFU tanh). Four packed multiplies or FMAs per two scores and no MUFU operation, which leaves the MUFU pipe
// to the exponentials.
constexpr float kCapPolyRange = 0.5f;
constexpr float kTanhP0 = 0x1.ffffeep-1f, kTanhP1 = -0x1.5542f2p-2f, kTanhP2 = 0x1.0e2330p-3f,
                kTanhP3 = -0x1.6bbec2p-5f;
__device__ __forceinline__ float tanh_poly(float u) {
  const float v = u * u;
  return u * fmaf(fmaf(fmaf(kTanhP3, v, kTanhP2), v, kTanhP1), v, kTanhP0);
}
// The same polynomial with the factor k = scale / cap folded into its coefficients, applied to the raw score z:
// tanh(k z) = z * sum_i (P_i k^(2i+1)) (z^2)^i. cf holds the four folded coefficients (packed pairs).
struct CapPoly {
  uint64_t c0, c1, c2, c3;
};
__device__ __forceinline__ CapPoly cap_poly_coeffs(float k) {
  const float k2 = k * k;
  const float c0 = kTanhP0 * k, c1 = kTanhP1 * k * k2, c2 = kTanhP2 * k * k2 * k2, c3 = kTanhP3 * k * k2 * k2 * k2;
  return CapPoly{f2_pack(c0, c0), f2_pack(c1, c1), f2_pack(c2, c2), f2_pack(c3, c3)};
}
__device__ __forceinline__ void cap_poly_pass(uint32_t (&zr)[BN], const CapPoly& cf) {
#pragma unroll
  for (int c = 0; c < BN; c += 2) {
    const uint64_t z = f2_pack(__uint_as_float(zr[c]), __uint_as_float(zr[c + 1]));
    const uint64_t v = f2_mul(z, z);
    const uint64_t p = f2_fma(f2_fma(f2_fma(cf.c3, v, cf.c2), v, cf.c1), v, cf.c0);
    float a, b;
    f2_unpack(f2_mul(p, z), a, b);
    zr[c] = __float_as_uint(a);
    zr[c + 1] = __float_as_uint(b);
  }
}

// Largest |z| of a row's 128 scores (8 independent partial maxima).
__device__ __forceinline__ float row_absmax(const uint32_t (&zr)[BN]) {
  float mx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mx[e] = fmaxf(fabsf(__uint_as_float(zr[2 * e])), fabsf(__uint_as_float(zr[2 * e + 1])));
#pragma unroll
  for (int c = 16; c < BN; c += 2)
    mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], fabsf(__uint_as_float(zr[c])), fabsf(__uint_as_float(zr[c + 1])));
  return fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
}

// Columns outside [lo_c, hi_c] (keys this row does not see) set to -inf: one unsigned compare per column.
__device__ __forceinline__ void mask_pass(uint32_t (&zr)[BN], int lo_c, int hi_c) {
  if (hi_c < lo_c) lo_c = BN, hi_c = BN;   // no visible column: c - lo_c wraps above the span for every c
  const uint32_t span = static_cast<uint32_t>(hi_c - lo_c);
#pragma unroll
  for (int c = 0; c < BN; ++c)
    zr[c] = static_cast<uint32_t>(c - lo_c) <= span ? zr[c] : __float_as_uint(-CUDART_INF_F);
}

// Row maximum: 8 independent partial maxima, two new scores per 3-input max.
__device__ __forceinline__ float row_max(const uint32_t (&zr)[BN]) {
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


// What the MMA issuer keeps of an item: tile ranges and the Q sequence numbers of its tiles.
struct IssItem {
  bool live;
  int tb0, te0, tb1, te1, tend;
  int q0, q1;   // Q tile sequence numbers (buffer = q % NQB)
};

// PAGED: keys come from a paged pool through the block table (a separate instantiation, so that the
// contiguous form carries none of the lookups).
template <bool PAGED, bool CAP>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmq,
                                                             const __grid_constant__ CUtensorMap tmk,
                                                             const __grid_constant__ CUtensorMap tmv,
                                                             const __grid_constant__ CUtensorMap tmo,
                                                             const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int window = prm.window;
  const int hpair = prm.hpair;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar = sbase + OFF_BAR;
  auto B = [&](int i) { return bar + 8u * i; };
  Item* ring = reinterpret_cast<Item*>(smem + OFF_ITEMS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < N_BARS; ++i) mbar_init(B(i), 1);
    for (int i = 0; i < NS; ++i) mbar_init(B(B_FU + i), 2);
    for (int w = 0; w < NQT; ++w) mbar_init(B(B_PF + w), BM);
    for (int i = 0; i < NI; ++i) mbar_init(B(B_IE + i), kItemReaders);
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
  pdl_wait();   // the stream's previous kernel (the cache update) has finished writing q and the caches

  // Cache row of key `key` of an item's plane: contiguous caches number rows plane + key; paged pools look
  // the key's block up (a K/V box of kbox rows never straddles two blocks); -1 when the block is missing.
  const KvLayout kvl = kv_layout(prm);
  auto key_row = [&](int plane, int key) -> int {
    if constexpr (!PAGED) return plane + key;
    const int row = plane / prm.hkv, g = plane - row * prm.hkv;
    const long long s = kv_slot(kvl, row, key);
    return s < 0 ? -1 : static_cast<int>(s + static_cast<long long>(g) * prm.block_size);
  };
  // One 128-key K or V tile (two 64-column halves, 128-byte swizzled) from boxes of kbox key rows, armed on
  // `bar` for the bytes it copies. A box without a block that lies wholly before the item's first visible
  // key (a pool that recycles out-of-window blocks) or wholly past the row's last key is skipped: its keys
  // are masked for every query of the item and the softmax warps zero its V rows. Any other missing block
  // is reported and read from row 0, so that the copy still delivers the bytes its barrier expects.
  // tile_rows looks the boxes up (paged pools: a block-table read each), issue_tile copies them; a producer
  // looks a tile up before it waits for the ring slot, so the table reads overlap that wait.
  struct TileRows {
    int r[BN / 64];
  };
  auto tile_rows = [&](int plane, int key, int first_vis, int kv_len) -> TileRows {
    TileRows t;
    if constexpr (!PAGED) {
      t.r[0] = plane + key;
    } else {
      for (int j = 0, b = 0; j < BN; j += prm.kbox, ++b) {
        t.r[b] = key_row(plane, key + j);
        if (t.r[b] < 0 && key + j + prm.kbox > first_vis && key + j < kv_len) {
          set_error(prm.err, kErrIndex);
          t.r[b] = 0;
        }
      }
    }
    return t;
  };
  auto issue_tile = [&](uint32_t dst, const CUtensorMap* tm, uint32_t bar, const TileRows& t) {
    if constexpr (!PAGED) {
      mbar_arrive_expect_tx(bar, TILE);
      tma_load_2d(dst, tm, bar, 0, t.r[0]);
      tma_load_2d(dst + HALF, tm, bar, 64, t.r[0]);
    } else {
      uint32_t bytes = 0;
      for (int j = 0, b = 0; j < BN; j += prm.kbox, ++b)
        if (t.r[b] >= 0) bytes += prm.kbox * 2 * 128;
      mbar_arrive_expect_tx(bar, bytes);
      for (int j = 0, b = 0; j < BN; j += prm.kbox, ++b) {
        if (t.r[b] < 0) continue;
        tma_load_2d(dst + j * 128, tm, bar, 0, t.r[b]);
        tma_load_2d(dst + HALF + j * 128, tm, bar, 64, t.r[b]);
      }
    }
  };
  // first key any query of an item sees (keys before it are masked for all of its rows)
  auto first_visible = [&](const Item& it) { return window > 0 ? max(0, it.fp + it.q0 - window + 1) : 0; };

  // item-ring reader (one thread): waits for entry e, copies it, releases it
  auto get_item = [&](int e, Item& it) -> bool {
    const int slot = e % NI;
    if (!mbar_wait(B(B_IF + slot), (e / NI) & 1, prm.err)) return false;
    it = ring[slot];
    mbar_arrive(B(B_IE + slot));
    return true;
  };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CTRL));
    if (warp == 11) {
      // ---------------------------------------------------------------- schedule (whole warp)
      // Items are the (chunk, q-tile) pairs times the query heads. The pairs are ranked by key-tile count,
      // heaviest first, ties in numbering order (pair p = y * n_seqs + chunk, y counting q-tiles from each
      // chunk's last); pairs without rows are dropped. Every CTA builds the same table, so the snake over
      // its ranks hands each item to exactly one CTA. The costs and counters live in the output staging
      // area, which no epilogue touches before this warp has published its first item. Batches with more
      // pairs (or larger costs) than the table holds keep the numbering order.
      uint16_t* order = reinterpret_cast<uint16_t*>(smem + OFF_ORD);
      int n_live = -1;   // pairs in the table; -1: no table
      const int n_pairs = prm.n_qt * prm.n_seqs;
      if (n_pairs <= kMaxPairs) {
        int* cost = reinterpret_cast<int*>(smem + OFF_E);
        int* bin = cost + kMaxPairs;   // bin b: pairs of cost cmax - b, then the first rank they take
        int cmax = -1;
        // Each chunk's start, length, first position and row, read once: with at most 32 chunks lane s holds
        // chunk s's (one round of independent loads, then shuffles), else every lane reads its pairs' own. The
        // table is the first thing every CTA waits for, so its loads are not left to run one after another.
        const bool few = prm.n_seqs <= 32;
        int m_q0 = 0, m_q1 = 0, m_fp = 0, m_row = 0;
        if (few && lane < prm.n_seqs) {
          m_q0 = prm.q_start[lane];
          m_q1 = prm.q_start[lane + 1];
          m_fp = prm.first_pos[lane];
          m_row = prm.rows[lane];
        }
        for (int p0 = 0; p0 < n_pairs; p0 += 32) {   // uniform trip count: the shuffles below take every lane
          const int p = p0 + lane;
          const int y = p / prm.n_seqs, s = p - y * prm.n_seqs;
          int q_a, q_b, fp, row;
          if (few) {
            const int src = p < n_pairs ? s : 0;
            q_a = __shfl_sync(0xffffffffu, m_q0, src);
            q_b = __shfl_sync(0xffffffffu, m_q1, src);
            fp = __shfl_sync(0xffffffffu, m_fp, src);
            row = __shfl_sync(0xffffffffu, m_row, src);
          } else if (p < n_pairs) {
            q_a = prm.q_start[s];
            q_b = prm.q_start[s + 1];
            fp = prm.first_pos[s];
            row = prm.rows[s];
          }
          if (p >= n_pairs) continue;
          Item it;
          it.n_b = q_b - q_a;
          it.q0 = (prm.n_qt - 1 - y) * (hpair ? BM : NQT * BM);
          it.fp = fp;
          int c = -1;
          if (it.q0 < it.n_b) {
            const bool bad = row < 0 || row >= prm.num_rows || it.fp < 0 || it.fp + it.n_b > prm.max_len;
            c = bad ? 0 : tiles_of(it, window, hpair).n;
          }
          cost[p] = c;
          cmax = max(cmax, c);
        }
        for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
        const int nb = cmax + 1;
        if (nb <= kMaxCostBins) {
          for (int b = lane; b < nb; b += 32) bin[b] = 0;
          __syncwarp();
          for (int p = lane; p < n_pairs; p += 32)
            if (cost[p] >= 0) atomicAdd(&bin[cmax - cost[p]], 1);
          __syncwarp();
          int carry = 0;   // exclusive scan of the counts: first rank of each bin
          for (int b0 = 0; b0 < nb; b0 += 32) {
            const int b = b0 + lane;
            const int v = b < nb ? bin[b] : 0;
            int incl = v;
            for (int o = 1; o < 32; o <<= 1) {
              const int t = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += t;
            }
            if (b < nb) bin[b] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
          }
          __syncwarp();
          n_live = carry;
          for (int p0 = 0; p0 < n_pairs; p0 += 32) {   // stable placement, 32 pairs at a time
            const int p = p0 + lane;
            const int c = p < n_pairs ? cost[p] : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, c);
            const int before = __popc(peers & ((1u << lane) - 1u));
            const int first = c >= 0 ? bin[cmax - c] : 0;
            __syncwarp();
            if (c >= 0) {
              order[first + before] = static_cast<uint16_t>(p);
              if (before == 0) bin[cmax - c] = first + __popc(peers);
            }
            __syncwarp();
          }
        }
      }
      __syncwarp();
      // ---------------------------------------------------------------- item decoder (lane 0)
      if (lane == 0) {
        const int hpu = hpair ? prm.hq / 2 : prm.hq;   // items per (chunk, q-tile) pair
        const int n_sched = n_live >= 0 ? n_live * hpu : prm.n_items;
        int e = 0, rounds = 0;
        bool ok = true;
        auto released = [&](int k) {   // wait until every reader has released entry k
          return mbar_wait(B(B_IE + k % NI), (k / NI) & 1, prm.err);
        };
        auto put = [&](const Item& it) -> bool {
          const int slot = e % NI;
          if (e >= NI && !released(e - NI)) return false;
          ring[slot] = it;
          mbar_arrive(B(B_IF + slot));   // release: the entry's stores are visible to the acquiring readers
          ++e;
          return true;
        };
        for (int r = 0; ok && r * G < n_sched && !*vabort; ++r) {
          const int id = item_of(r, cta, G);
          if (id >= n_sched) continue;
          const int pr = id / hpu, h = (id - pr * hpu) << hpair;
          const int p = n_live >= 0 ? order[pr] : pr;
          const int y = p / prm.n_seqs, s = p - y * prm.n_seqs;
          Item it;
          it.t0 = prm.q_start[s];
          it.n_b = prm.q_start[s + 1] - it.t0;
          it.q0 = (prm.n_qt - 1 - y) * (hpair ? BM : NQT * BM);
          if (it.q0 >= it.n_b) continue;           // this chunk has no rows that far
          const int row = prm.rows[s];
          it.fp = prm.first_pos[s];
          it.h = h;
          const bool bad = row < 0 || row >= prm.num_rows || it.fp < 0 || it.fp + it.n_b > prm.max_len;
          it.kind = bad ? kBad : kLive;
          it.plane = bad ? 0 : (row * prm.hkv + h / (prm.hq / prm.hkv)) * (PAGED ? 1 : prm.max_len);
          it.round0 = rounds;
          if (!bad) rounds += tiles_of(it, window, hpair).n;
          ok = put(it);
        }
        if (ok) {
          Item end;
          end.kind = kEnd;
          end.t0 = end.n_b = end.q0 = end.fp = end.plane = end.h = 0;
          end.round0 = rounds;
          ok = put(end);
        }
        if (!ok) abort_flag = 1;
      }
    } else if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer: Q tiles, K halves
      // Ring slot j holds the K tile of global round j (the tile the scores issued in round j - 1 use) and
      // the V tile of round j - 1; this producer fills the K halves (the last slot has none: a bare
      // arrival). Per item: Q0, the first K tile, Q1, the remaining K tiles.
      prefetch_tmap(&tmq);
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
      int qn = 0, kj = 0;   // Q tiles loaded, ring slots filled
      bool ok = true;
      auto load_q = [&](const Item& it, int w) -> bool {
        const int b = qn % NQB, u = qn / NQB;
        if (u > 0 && !mbar_wait(B(B_QE + b), (u - 1) & 1, prm.err)) return false;
        const int tok = it.t0 + qt_row(it, w, hpair), hd = qt_head(it, w, hpair);
        mbar_arrive_expect_tx(B(B_QF + b), TILE);
        tma_load_3d(sbase + OFF_Q + b * TILE, &tmq, B(B_QF + b), 0, hd, tok);
        tma_load_3d(sbase + OFF_Q + b * TILE + HALF, &tmq, B(B_QF + b), 64, hd, tok);
        ++qn;
        return true;
      };
      auto fill_k = [&](int plane, int key, int first_vis, int kv_len) -> bool {   // plane < 0: no K tile
        const int st = kj % NS;
        TileRows rows{};
        if (plane >= 0) rows = tile_rows(plane, key, first_vis, kv_len);
        if (kj >= NS && !mbar_wait(B(B_EM + st), ((kj / NS) - 1) & 1, prm.err)) return false;
        if (plane >= 0) {
          issue_tile(sbase + OFF_R + st * 2 * TILE, &tmk, B(B_FU + st), rows);
        } else {
          mbar_arrive(B(B_FU + st));
        }
        ++kj;
        return true;
      };
      // The next item's Q tiles and first K/V tiles are fetched into L2 when this item starts: its Q buffers
      // free only about one round before the tensor core needs them, too late for a DRAM round trip.
      auto prefetch_next = [&](int e) -> bool {
        const int slot = e % NI;
        if (!mbar_wait(B(B_IF + slot), (e / NI) & 1, prm.err)) return false;
        const Item& nx = ring[slot];   // read without releasing: get_item(e) releases it later
        if (nx.kind != kLive) return true;
        const Tiles T = tiles_of(nx, window, hpair);
        for (int w = 0; w < (T.valid1 ? 2 : 1); ++w) {
          const int tok = nx.t0 + qt_row(nx, w, hpair), hd = qt_head(nx, w, hpair);
          tma_prefetch_3d(&tmq, 0, hd, tok);
          tma_prefetch_3d(&tmq, 64, hd, tok);
        }
        // (paged pools: Q only; the block-table read that the first K/V box needs would hold this producer
        // up for longer than the prefetch saves)
        const int key = PAGED ? -1 : key_row(nx.plane, first_visible(nx) / prm.kbox * prm.kbox);
        if (key >= 0) {
          tma_prefetch_2d(&tmk, 0, key);
          tma_prefetch_2d(&tmk, 64, key);
          tma_prefetch_2d(&tmv, 0, key);
          tma_prefetch_2d(&tmv, 64, key);
        }
        return true;
      };
      for (int e = 0; ok; ++e) {
        Item it;
        if (!get_item(e, it)) { ok = false; break; }
        if (it.kind == kEnd) break;
        if (!prefetch_next(e + 1)) { ok = false; break; }
        if (it.kind != kLive) continue;
        const Tiles T = tiles_of(it, window, hpair);
        if (!load_q(it, 0)) { ok = false; break; }
        for (int i = 0; ok && i < T.n; ++i) {
          if (*vabort || (i == 1 && T.valid1 && !load_q(it, 1)) ||
              !fill_k(it.plane, (T.tb0 + i) * BN, first_visible(it), it.fp + it.n_b))
            ok = false;
        }
        if (ok && T.n == 1 && T.valid1 && !load_q(it, 1)) ok = false;
      }
      if (ok && !fill_k(-1, 0, 0, 0)) ok = false;
      if (!ok) abort_flag = 1;
      // every issued copy must land before the CTA's shared memory is released
      for (int j = max(0, qn - NQB); j < qn; ++j) mbar_wait(B(B_QF + j % NQB), (j / NQB) & 1, prm.err);
      for (int j = max(0, kj - NS); j < kj; ++j) mbar_wait(B(B_FU + j % NS), (j / NS) & 1, prm.err);
    } else if (warp == 10 && lane == 0) {
      // ---------------------------------------------------------------- TMA producer: V halves
      // slot 0 has no V tile (a bare arrival); slot j > 0 holds the V tile of global round j - 1
      prefetch_tmap(&tmv);
      int vj = 0;
      bool ok = true;
      auto fill_v = [&](int plane, int key, int first_vis, int kv_len) -> bool {   // plane < 0: no V tile
        const int st = vj % NS;
        TileRows rows{};
        if (plane >= 0) rows = tile_rows(plane, key, first_vis, kv_len);
        if (vj >= NS && !mbar_wait(B(B_EM + st), ((vj / NS) - 1) & 1, prm.err)) return false;
        if (plane >= 0) {
          issue_tile(sbase + OFF_R + st * 2 * TILE + TILE, &tmv, B(B_FU + st), rows);
        } else {
          mbar_arrive(B(B_FU + st));
        }
        ++vj;
        return true;
      };
      ok = fill_v(-1, 0, 0, 0);
      for (int e = 0; ok; ++e) {
        Item it;
        if (!get_item(e, it)) { ok = false; break; }
        if (it.kind == kEnd) break;
        if (it.kind != kLive) continue;
        const Tiles T = tiles_of(it, window, hpair);
        for (int i = 0; ok && i < T.n; ++i) {
          if (*vabort || !fill_v(it.plane, (T.tb0 + i) * BN, first_visible(it), it.fp + it.n_b)) ok = false;
        }
      }
      if (!ok) abort_flag = 1;
      for (int j = max(0, vj - NS); j < vj; ++j) mbar_wait(B(B_FU + j % NS), (j / NS) & 1, prm.err);
    } else if (warp == 9 && lane == 0) {
      // ---------------------------------------------------------------- MMA issuer (one thread)
      // Rounds run over all items' key tiles in order. Round (tile t of item A, next tile u: t + 1, or the
      // first tile of the next item B after A's last) reads ring slot g + 1 (V(t), K(u)):
      //   PV0(t), S0(u), PV1(t), S1(u), release of the slot.
      // Each tcgen05.mma blocks the issuing thread until the tensor core takes it (the queue is short),
      // so every wait between two MMA groups idles the tensor core: the operand waits (the slot, a Q tile)
      // sit at the top of the round, and between groups there are only the P waits. A Q buffer is
      // released by a commit after the last scores that read it.
      int qseq = 0, e = 0;
      bool ok = true, ended = false;   // ended: the end-of-list entry has been read
      auto next_live = [&](IssItem& I) {
        I.live = false;
        while (ok && !ended) {
          Item it;
          if (!get_item(e, it)) { ok = false; return; }
          ++e;
          if (it.kind == kEnd) {
            ended = true;
            return;
          }
          if (it.kind != kLive) continue;
          const Tiles T = tiles_of(it, window, hpair);
          I.live = true;
          I.tb0 = T.tb0;
          I.te0 = T.te0;
          I.tb1 = T.tb1;
          I.te1 = T.te1;
          I.tend = T.tb0 + T.n - 1;
          I.q0 = qseq;
          I.q1 = qseq + 1;
          qseq += T.valid1 ? 2 : 1;
          return;
        }
      };
      auto qready = [&](int q) { return mbar_wait(B(B_QF + q % NQB), (q / NQB) & 1, prm.err); };
      auto qsmem = [&](int q) { return sbase + OFF_Q + (q % NQB) * TILE; };
      IssItem A, Bn;
      next_live(A);
      next_live(Bn);
      int st = 0, ph = 0;        // ring slot of the next round: stage, phase
      int npv0 = 0, npv1 = 0;    // PVs issued per stream (phase of p_full)
      bool a_q1 = false, b_q1 = false;   // Q1 of A / of B waited on
      if (ok && A.live) {
        // scores of A's first tile, from ring slot 0
        ok = mbar_wait(B(B_FU), 0, prm.err) && qready(A.q0);
        if (ok) {
          tc_fence_after();
          issue_s(tmem, qsmem(A.q0), sbase + OFF_R);
          tc_commit(B(B_SF + 0));
          if (A.te0 == A.tb0) tc_commit(B(B_QE + A.q0 % NQB));
          if (A.tb1 <= A.tb0 && A.tb0 <= A.te1) {
            ok = qready(A.q1);
            a_q1 = true;
            if (ok) {
              issue_s(tmem + BN, qsmem(A.q1), sbase + OFF_R);
              tc_commit(B(B_SF + 1));
              if (A.te1 == A.tb0) tc_commit(B(B_QE + A.q1 % NQB));
            }
          }
          tc_commit(B(B_EM + 0));
          st = 1 % NS;
          ph = (1 / NS) & 1;
        }
      }
      while (ok && A.live) {
        bool first0 = true, first1 = true;
        const uint32_t q0s = qsmem(A.q0), q1s = qsmem(A.q1);
        // PVs of tile t (the P waits are the only waits between MMA groups)
        auto pv0 = [&](int t, uint32_t vs) -> bool {
          if (!mbar_wait(B(B_PF + 0), npv0 & 1, prm.err)) return false;
          tc_fence_after();
          issue_pv(tmem + 256, tmem, vs, !first0);
          first0 = false;
          ++npv0;
          if (t == A.te0) tc_commit(B(B_OD + 0));   // Q0's output is final
          return true;
        };
        auto pv1 = [&](int t, uint32_t vs) -> bool {
          if (!mbar_wait(B(B_PF + 1), npv1 & 1, prm.err)) return false;
          tc_fence_after();
          issue_pv(tmem + 256 + D, tmem + BN, vs, !first1);
          first1 = false;
          ++npv1;
          if (t == A.te1) tc_commit(B(B_OD + 1));   // Q1's output is final
          return true;
        };
        // rounds inside the item: the next tile u = t + 1 is the item's own
        for (int t = A.tb0; ok && t < A.tend; ++t) {
          const int u = t + 1;
          const bool s0u = u <= A.te0, s1u = A.tb1 <= u && u <= A.te1;
          const uint32_t ks = sbase + OFF_R + st * 2 * TILE, vs = ks + TILE;
          if (!mbar_wait(B(B_FU + st), ph, prm.err)) { ok = false; break; }
          if (s1u && !a_q1) {
            if (!qready(A.q1)) { ok = false; break; }
            a_q1 = true;
          }
          if (t <= A.te0 && !pv0(t, vs)) { ok = false; break; }
          if (s0u) {
            issue_s(tmem, q0s, ks);
            tc_commit(B(B_SF + 0));
            if (u == A.te0) tc_commit(B(B_QE + A.q0 % NQB));
          }
          if (t >= A.tb1 && t <= A.te1 && !pv1(t, vs)) { ok = false; break; }
          if (s1u) {
            issue_s(tmem + BN, q1s, ks);
            tc_commit(B(B_SF + 1));
            if (u == A.te1) tc_commit(B(B_QE + A.q1 % NQB));
          }
          tc_commit(B(B_EM + st));
          if (++st == NS) {
            st = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        {
          // the item's last round: the next tile is the first of the next item (its Q tiles waited here)
          const int t = A.tend, u = Bn.tb0;
          const bool s0u = Bn.live, s1u = Bn.live && Bn.tb1 <= u && u <= Bn.te1;
          const uint32_t ks = sbase + OFF_R + st * 2 * TILE, vs = ks + TILE;
          if (*vabort || !mbar_wait(B(B_FU + st), ph, prm.err) || (s0u && !qready(Bn.q0))) {
            ok = false;
            break;
          }
          b_q1 = s1u;
          if (t <= A.te0 && !pv0(t, vs)) { ok = false; break; }
          if (s0u) {
            issue_s(tmem, qsmem(Bn.q0), ks);
            tc_commit(B(B_SF + 0));
            if (u == Bn.te0) tc_commit(B(B_QE + Bn.q0 % NQB));
          }
          if (t >= A.tb1 && t <= A.te1 && !pv1(t, vs)) { ok = false; break; }
          if (s1u) {
            // Bn's Q1 reuses A's Q1 buffer, freed by the S1 issued in the round before: waited on last
            if (!qready(Bn.q1)) { ok = false; break; }
            issue_s(tmem + BN, qsmem(Bn.q1), ks);
            tc_commit(B(B_SF + 1));
            if (u == Bn.te1) tc_commit(B(B_QE + Bn.q1 % NQB));
          }
          tc_commit(B(B_EM + st));
          if (++st == NS) {
            st = 0;
            ph ^= 1;
          }
        }
        A = Bn;
        a_q1 = b_q1;
        b_q1 = false;
        next_live(Bn);
      }
      if (!ok) abort_flag = 1;
      tc_commit(B(B_DR));
      mbar_wait(B(B_DR), 0, prm.err);   // all MMAs done before TMEM may be released
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
    // ---------------------------------------------------------------- softmax (8 warps, 1 row each thread)
    const int w = warp >> 2;             // which Q tile
    const int wi = warp & 3;             // TMEM lane quarter
    const int r = wi * 32 + lane;        // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(wi * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + w * BN;
    const uint32_t t_o = tmem + lane_addr + 256 + w * D;
    const float cap = CAP ? prm.softcap : 0.f;   // uncapped layers run an instantiation without the cap code
    const float cap_in = cap > 0.f ? prm.scale / cap : 0.f;
    const CapPoly cap_cf = cap_poly_coeffs(cap_in);
    // z * zmul is the logit in log2 units: z the raw score, or for capped layers tanh(scale z / cap)
    const float zmul = cap > 0.f ? cap * kLog2e : prm.scale * kLog2e;
    int ns = 0, nod = 0;
    bool ok = true;
    // The epilogue of an item (O / l out through the warp's staging slot) is deferred into the first tile
    // of this warpgroup's next item: that tile's softmax runs first (it does not touch O), then O is read
    // from TMEM just before the P arrival that lets the next PV overwrite it, and the stores go out while
    // the tensor core runs that PV. The finished item's ring entry is held until then; its fields are read
    // back from shared memory.
    bool pend = false;      // an epilogue is pending
    int pend_slot = 0;      // its item's ring entry
    float pend_inv_l = 0.f; // its row's 1 / l
    // O / l of the pending item -> pw (bf16 pairs)
    auto epi_read = [&](uint32_t (&pw)[D / 2]) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(B(B_OD + w), nod & 1, prm.err))) return false;
      ++nod;
      tc_fence_after();
      {
        uint32_t ov[D];   // the whole O row in one tensor-memory load and one wait
        tmem_ld128(t_o, ov);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 2; ++c)
          pw[c] = pack_bf16(__uint_as_float(ov[2 * c]) * pend_inv_l, __uint_as_float(ov[2 * c + 1]) * pend_inv_l);
      }
      tc_fence_before();   // O_w has been read
      return true;
    };
    // Two groups of 16 rows per warp: the group's lanes write their rows into the warp's staging slot in the
    // 128-byte-swizzled layout (two 64-wide halves) and lane 0 stores them with two TMA tensor stores; a
    // group whose rows run past the chunk stores row by row instead (a whole box would overwrite the next
    // chunk's rows). Then the pending item's ring entry is released.
    auto epi_store = [&](const uint32_t (&pw)[D / 2]) {
      const Item& pi = ring[pend_slot];
      const int t0 = pi.t0, n_b = pi.n_b, h = qt_head(pi, w, hpair);
      const int row0 = qt_row(pi, w, hpair) + wi * 32;   // chunk row of this warp's lane 0
      mbar_arrive(B(B_IE + pend_slot));
      uint8_t* stg = smem + OFF_E + warp * STG;
      const uint32_t stg_a = sbase + OFF_E + warp * STG;
      const int rr = lane & 15;
#pragma unroll
      for (int hg = 0; hg < 2; ++hg) {
        const int g0 = row0 + hg * 16;
        const bool mine = (lane >> 4) == hg;
        if (g0 + 16 <= n_b) {
          if (mine) {
#pragma unroll
            for (int c16 = 0; c16 < 16; ++c16)
              *reinterpret_cast<uint4*>(stg + (c16 >> 3) * (STG / 2) + rr * 128 + (((c16 & 7) ^ (rr & 7)) << 4)) =
                  make_uint4(pw[4 * c16], pw[4 * c16 + 1], pw[4 * c16 + 2], pw[4 * c16 + 3]);
          }
          fence_proxy_async_smem();          // generic-proxy writes -> visible to the copy engine
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmo, stg_a, 0, h, t0 + g0);
            tma_store_3d(&tmo, stg_a + STG / 2, 64, h, t0 + g0);
            bulk_commit();
            bulk_wait_read();                // the slot is rewritten by the next group
          }
          __syncwarp();
        } else if (mine && g0 + rr < n_b) {
          uint4* orow = reinterpret_cast<uint4*>(prm.out + (static_cast<long long>(t0 + g0 + rr) * prm.hq + h) * D);
#pragma unroll
          for (int c16 = 0; c16 < 16; ++c16)
            orow[c16] = make_uint4(pw[4 * c16], pw[4 * c16 + 1], pw[4 * c16 + 2], pw[4 * c16 + 3]);
        }
      }
    };
    // A pending epilogue is flushed at once on an item this warpgroup takes no part in (nothing overwrites
    // its O there), so that its ring entry is never held across several items.
    auto flush = [&]() {
      if (!pend) return;
      uint32_t pw[D / 2];
      if (epi_read(pw)) epi_store(pw);
      else ok = false;
      pend = false;
    };
    for (int e = 0; ok; ++e) {
      const int slot = e % NI;
      if (!__all_sync(0xffffffffu, mbar_wait(B(B_IF + slot), (e / NI) & 1, prm.err))) {
        abort_flag = 1;
        break;
      }
      const Item& it = ring[slot];
      const int kind = it.kind;
      int my_tb = 0, my_te = -1, my_pmin = 0, my_pmax = 0, kv_len = 0;
      if (kind == kLive) {
        const Item itc = it;
        const Tiles T = tiles_of(itc, window, hpair);
        if (w == 0 || T.valid1) {
          my_tb = w == 0 ? T.tb0 : T.tb1;
          my_te = w == 0 ? T.te0 : T.te1;
          my_pmin = w == 0 ? T.pmin0 : T.pmin1;
          my_pmax = w == 0 ? T.pmax0 : T.pmax1;
          kv_len = itc.fp + itc.n_b;
        }
      }
      if (my_te < my_tb) {
        // an entry this warpgroup takes no part in: the end of the list, a chunk whose rows the tables place
        // outside the cache (zero outputs, error word set, nothing loaded), or an item without this Q tile
        flush();
        if (kind == kBad) {
          const int qrow = qt_row(it, w, hpair) + r;
          if (w == 0 && r == 0) set_error(prm.err, kErrIndex);
          if (qrow < it.n_b) {
            uint4* o = reinterpret_cast<uint4*>(
                prm.out + (static_cast<long long>(it.t0 + qrow) * prm.hq + qt_head(it, w, hpair)) * D);
#pragma unroll
            for (int j = 0; j < D / 8; ++j) o[j] = make_uint4(0, 0, 0, 0);
          }
        }
        mbar_arrive(B(B_IE + slot));
        if (kind == kEnd) break;
        continue;
      }
      const int p = my_pmin + r;         // this row's position
      float m = -CUDART_INF_F, l = 0.f;
      int nact = 0;
      for (int t = my_tb; t <= my_te; ++t) {
        // outcomes are made warp-uniform: the TMEM loads and stores below are warp-collective
        if (__any_sync(0xffffffffu, *vabort != 0)) { ok = false; break; }
        if (!__all_sync(0xffffffffu, mbar_wait(B(B_SF + w), ns & 1, prm.err))) {
          abort_flag = 1;
          ok = false;
          break;
        }
        ++ns;
        tc_fence_after();
        uint32_t zr[BN];
        tmem_ld128(t_s, zr);
        tmem_wait_ld();
        const int kstart = t * BN;
        const bool need_mask = !(kstart + BN - 1 <= my_pmin &&
                                 (window == 0 || my_pmax - kstart <= window - 1) && kstart + BN <= kv_len);
        // zr: the raw score q.k, or for capped layers tanh(scale q.k / cap); either way zr * zmul is the logit
        // in log2 units (the factor is applied inside the exponent). Visible keys: columns [lo_c, hi_c].
        const int hi_c = min(p, kv_len - 1) - kstart;
        const int lo_c = window > 0 ? p - window + 1 - kstart : -BN;
        float tmax, amax = 0.f;
        bool poly = false;
        if (!PAGED && cap > 0.f && !need_mask) {   // (the paged form has no registers to spare for it)
          amax = row_absmax(zr);
          poly = __all_sync(0xffffffffu, amax * cap_in <= kCapPolyRange);
        }
        if (poly) {
          // every score of the warp's rows is small: the FMA-pipe tanh; the tile max is bounded by the cap of
          // the row's largest |z| (an upper bound of its capped logits is all the online softmax needs: the
          // exponents stay within 2 * cap * tanh(0.5) of it, far from underflow)
          cap_poly_pass(zr, cap_cf);
          tmax = tanh_poly(amax * cap_in) * zmul;
        } else {
          if (cap > 0.f) cap_pass(zr, cap_in);
          if (need_mask) mask_pass(zr, lo_c, hi_c);
          tmax = row_max(zr) * zmul;
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
        // keys before lo_zero: boxes a paged pool may have recycled (not loaded when their block is gone)
        const int lo_zero = (PAGED && prm.kbox < BN) ? first_visible(it) : 0;
        if (kstart + BN > kv_len || kstart < lo_zero) {
          // V rows past the row's last key hold whatever the cache holds there (maybe NaN), and rows of a
          // skipped box whatever the stage held before; P is 0 there, but 0 * NaN is NaN, so zero those rows
          // before the tensor core reads them (after the V copy has landed; the stage cannot be refilled
          // before this tile's PV, which waits for us).
          const int tb0 = first_visible(it) / BN;   // the item's first tile
          const int g = it.round0 + t - tb0 + 1;   // ring slot of this tile's round
          if (!__all_sync(0xffffffffu, mbar_wait(B(B_FU + g % NS), (g / NS) & 1, prm.err))) {
            abort_flag = 1;
            ok = false;
            break;
          }
          if (kstart + r >= kv_len || kstart + r < lo_zero) {
            uint8_t* vtile = smem + OFF_R + (g % NS) * 2 * TILE + TILE;   // V(t), in the round slot of tile t
            uint4* vrow0 = reinterpret_cast<uint4*>(vtile + r * 128);
            uint4* vrow1 = reinterpret_cast<uint4*>(vtile + HALF + r * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              vrow0[c] = make_uint4(0, 0, 0, 0);
              vrow1[c] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        if (pend) {
          // the previous item's O is read before this P lets the next PV overwrite it
          uint32_t pw[D / 2];
          if (!epi_read(pw)) {
            abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive(B(B_PF + w));
          epi_store(pw);
          pend = false;
        } else {
          mbar_arrive(B(B_PF + w));
        }
        ++nact;
      }
      if (!ok) break;
      pend = true;                        // this item's epilogue: deferred (its ring entry stays held)
      pend_slot = slot;
      if (prm.sinks) l += ex2(prm.sinks[qt_head(it, w, hpair)] * kLog2e - m);   // one more logit, no value
      pend_inv_l = l > 0.f ? 1.f / l : 0.f;
    }
    if (!ok) abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace pf

template <bool PAGED, bool CAP>
static cudaError_t run_prefill(const CUtensorMap& tmq, const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const CUtensorMap& tmo, const pf::Params& prm, int grid, cudaStream_t stream) {
  using namespace pf;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<PAGED, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_dependent(prefill_kernel<PAGED, CAP>, dim3(grid), dim3(THREADS), SMEM_BYTES, stream, tmq, tmk, tmv,
                          tmo, prm);
}

cudaError_t launch_prefill_bf16(const AttnArgs& a, cudaStream_t stream) {
  using namespace pf;
  if (a.n_seqs == 0 || a.max_q_len == 0 || a.n_tokens == 0) return cudaSuccess;
  CUtensorMap tmq, tmk, tmv, tmo;
  const uint64_t rows_total = a.block_table ? static_cast<uint64_t>(a.n_blocks) * a.hkv * a.block_size
                                            : static_cast<uint64_t>(a.num_rows) * a.hkv * a.max_len;
  const int kbox = (a.block_table && a.block_size % BN != 0) ? 64 : BN;   // pools: block sizes are multiples of 64
  // q_rot and out [N, Hq, D]: q rows past N are zero-filled by the copy engine, never read from memory; out
  // boxes (16 rows) are only stored whole when all their rows belong to the chunk
  const uint64_t n_tok = static_cast<uint64_t>(a.n_tokens);
  if (!encode_tmap_3d_bf16(&tmq, a.q_rot, D, a.hq, n_tok, D * 2, static_cast<uint64_t>(a.hq) * D * 2, 64, 1, BM) ||
      !encode_tmap_3d_bf16(&tmo, a.out, D, a.hq, n_tok, D * 2, static_cast<uint64_t>(a.hq) * D * 2, 64, 1, 16) ||
      !encode_tmap_2d_bf16(&tmk, a.k_cache, D, rows_total, D * 2, 64, kbox) ||
      !encode_tmap_2d_bf16(&tmv, a.v_cache, D, rows_total, D * 2, 64, kbox))
    return cudaErrorInvalidValue;
  const int hpair = (a.hq / a.hkv) % 2 == 0 ? 1 : 0;
  const int item_rows = hpair ? BM : NQT * BM;
  const long long n_qt = (a.max_q_len + item_rows - 1) / item_rows;
  const long long n_items = n_qt * a.n_seqs * (hpair ? a.hq / 2 : a.hq);
  if (n_items > 0x3fffffffLL) return cudaErrorInvalidValue;
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
  prm.n_seqs = a.n_seqs;
  prm.n_qt = static_cast<int>(n_qt);
  prm.n_items = static_cast<int>(n_items);
  prm.hpair = hpair;
  prm.softcap = a.softcap;
  prm.sinks = a.sinks;
  prm.block_table = a.block_table;
  prm.block_size = a.block_size;
  prm.max_blocks = a.max_blocks;
  prm.n_blocks = a.n_blocks;
  prm.kbox = kbox;
  prm.scale = a.scale;
  prm.err = a.err;
  int dev = 0, n_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (shared memory and all 512 TMEM columns allow no second one)
  int grid = static_cast<int>(std::min<long long>(n_items, n_sm));
  if (a.max_ctas > 0) grid = std::min(grid, a.max_ctas);   // the rest of the SMs left to a concurrent decode
  const bool paged = a.block_table != nullptr, capped = a.softcap > 0.f;
  if (paged) {
    return capped ? run_prefill<true, true>(tmq, tmk, tmv, tmo, prm, grid, stream)
                  : run_prefill<true, false>(tmq, tmk, tmv, tmo, prm, grid, stream);
  }
  return capped ? run_prefill<false, true>(tmq, tmk, tmv, tmo, prm, grid, stream)
                : run_prefill<false, false>(tmq, tmk, tmv, tmo, prm, grid, stream);
}

}  // namespace da
