// Internal interface between the host API (api.cpp) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include "decattn.h"

namespace da {

constexpr int kMaxRotHalf = 128;  // r/2 <= 128 (r <= 256)

// Error flags ORed into the device error word (the word itself lives in errors.cu).
constexpr int kErrIndex = 1;
constexpr int kErrTimeout = 2;

int* error_word_ptr();
int read_and_clear_error_word(cudaStream_t stream, int* flags);

// Frequencies of one rope configuration, computed on the host in fp64. Tokens whose sequence length
// exceeds `switch_len` use the long table (LongRoPE); otherwise the short one. inv_* are the angular
// frequencies (radians per position); turn_* are the same frequencies in turns per position as 64-bit
// fixed-point fractions (value * 2^64), which the device multiplies by the integer position modulo 2^64:
// the wrap-around is the exact reduction of the angle modulo 2 pi.
struct RopeFreqs {
  int half;                      // r / 2
  int switch_len;                // long table when seq_len > switch_len; INT32_MAX when unused
  int use_seq_len;               // 1: read seq_len[] (LongRoPE)
  double af;                     // attention factor multiplying cos and sin
  double inv_short[kMaxRotHalf];
  double inv_long[kMaxRotHalf];
};
struct RopeTurns {
  int half, switch_len, use_seq_len;
  float af;
  unsigned long long turn_short[kMaxRotHalf];
  unsigned long long turn_long[kMaxRotHalf];
};
RopeTurns rope_turns(const RopeFreqs& f);

cudaError_t launch_rope_tables(const RopeFreqs& f, const int32_t* positions, const int32_t* seq_len, int n,
                               float* cos, float* sin, int* err, cudaStream_t stream);

// Where the cache slot of (row, KV head, position) lives. Contiguous caches [num_rows, Hkv, max_len, d]:
// block_table == NULL. Paged pools [n_blocks, Hkv, block_size, d]: position p of a row lives in block
// block_table[row * max_blocks + p / block_size] at offset p % block_size, and max_len = max_blocks *
// block_size.
struct KvLayout {
  const int32_t* block_table;
  int num_rows, max_len, hkv;
  int block_size, max_blocks, n_blocks;
};

struct KvUpdateArgs {
  const void* q;
  const void* k;
  const void* v;
  int n, hq, hkv, d, rot;
  const int32_t* rows;
  const int32_t* positions;
  const float* cos;
  const float* sin;
  const float* q_norm_w;
  const float* k_norm_w;
  float eps;
  void* q_rot;
  void* k_cache;
  void* v_cache;
  int num_rows, max_len;
  const int32_t* block_table;     // paged pool: [num_rows, max_blocks] block ids; NULL: contiguous cache
  int block_size, max_blocks, n_blocks;
  int* err;
  int wpt;                        // warps per token (set by the launcher)
  const int32_t* seq_len;         // per token, for LongRoPE's table switch (fused form only)
};
cudaError_t launch_kv_update(const KvUpdateArgs& a, bool bf16, cudaStream_t stream);
// The same update with each token's cos/sin formed in the kernel from its position (no tables); bf16, d 128,
// r/2 a multiple of 8. cos/sin in a are unused.
bool kv_update_rope_supported(bool bf16, int d, int rot);
cudaError_t launch_kv_update_rope(const KvUpdateArgs& a, const RopeFreqs& freqs, cudaStream_t stream);

// Query set of an attention call: prefill chunks (q_start/first_pos) or decode tokens (positions).
struct AttnArgs {
  const void* q_rot;
  const void* k_cache;
  const void* v_cache;
  void* out;
  int hq, hkv, d;
  int num_rows, max_len;
  int n_seqs;
  const int32_t* rows;
  const int32_t* q_start;         // prefill: [S+1]; NULL for decode (one token per sequence)
  const int32_t* first_pos;       // prefill: [S]
  const int32_t* positions;       // decode: [S]
  int max_q_len;                  // prefill: grid bound; decode: 1
  int n_tokens;                   // rows of q_rot/out (prefill: q_start[S]; decode: S)
  const int32_t* key_positions;   // [R, M] or NULL
  const int32_t* block_table;     // paged pool: [num_rows, max_blocks] block ids; NULL: contiguous cache
  int block_size, max_blocks, n_blocks;
  int window;
  float softcap;
  float scale;
  const float* sinks;             // [Hq] sink logits (natural units) or NULL
  int* err;
  int max_ctas;                   // tcgen05 prefill: at most this many persistent CTAs (0: one per SM)
};
cudaError_t launch_attn_generic(const AttnArgs& a, bool bf16, cudaStream_t stream);

// Split-K decode (bf16, d = 128, Hq/Hkv <= 8, no key_positions).
struct DecodePlan {
  int chunk;      // keys per split (multiple of 64; of 256 for 128 heads)
  int n_splits;   // splits per (sequence, KV head) at most
};
// aligned: chunks start at the window start rounded down to a 64-key tile (paged pools)
DecodePlan decode_plan(int hkv, int n_seqs, int max_len, int window, bool aligned);
size_t decode_workspace_bytes(int hq, int n_seqs, const DecodePlan& p);
cudaError_t launch_decode_bf16(const AttnArgs& a, const DecodePlan& p, void* workspace, cudaStream_t stream);

// Fixed scratch for da_attn_decode_noalloc (file-scope device array in attn_decode.cu).
constexpr size_t kDecodeStaticScratchBytes = size_t(32) << 20;
void* static_scratch();   // its device address on the current device; NULL if the lookup fails

// tcgen05 prefill (bf16, d = 128, no key_positions).
cudaError_t launch_prefill_bf16(const AttnArgs& a, cudaStream_t stream);

// MLA (latent rank 512, rotary 64, bf16): cache rows [num_rows, max_len, 576] or a paged pool of such rows.
struct MlaUpdateArgs {
  const void* latent;             // [n, 512]
  const void* k_rope;             // [n, 64], adjacent pairs
  const int32_t* rows;
  const int32_t* positions;
  const float* cos;               // [n, 32]
  const float* sin;
  void* q;                        // [n, Hq, 576] or NULL (rotary part rotated in place)
  void* cache;
  int n, hq, num_rows, max_len;
  const int32_t* block_table;     // paged pool or NULL
  int block_size, max_blocks, n_blocks;
  int* err;
};
struct MlaArgs {
  const void* q;                  // [S, Hq, 576]
  const void* cache;
  void* out;                      // [S, Hq, 512]
  int hq, num_rows, max_len, n_seqs, window;
  float scale;
  const int32_t* rows;
  const int32_t* positions;
  const int32_t* block_table;
  int block_size, max_blocks, n_blocks;
  int* err;
};
struct MlaPlan {
  int chunk;      // keys per split (multiple of 64; of 256 for 128 heads)
  int n_splits;
};
MlaPlan mla_plan(int hq, int n_seqs, int max_len, int window, bool aligned);
size_t mla_workspace_bytes(int hq, int n_seqs, const MlaPlan& p);
cudaError_t launch_mla_update(const MlaUpdateArgs& a, cudaStream_t stream);
cudaError_t launch_mla_decode(const MlaArgs& a, const MlaPlan& plan, void* workspace, cudaStream_t stream);
// 128-head layers: the tcgen05 CTA-pair kernel (chunks a multiple of 256 keys); partials in the same layout
int mla_pair_chunk(int n_seqs, int max_keys);
cudaError_t launch_mla_pair_decode(const MlaArgs& a, const MlaPlan& plan, float* ws_o, float2* ws_ml,
                                   cudaStream_t stream);

// Projections (tcgen05 GEMM, bf16, K a multiple of 64, N a multiple of 256): y = x w^T (+ bias), or with
// q_rot set, the stacked q/k/v projection with norm, RoPE (head_dim 128, all dims rotated) and cache write
// fused into the epilogue.
struct ProjArgs {
  const void* x;                  // [m, k]
  const void* w;                  // [n, k]
  const float* bias;              // [n] or NULL
  int m, n, k;
  void* y;                        // [m, n] (plain)
  int hq, hkv;
  const float* q_norm_w;
  const float* k_norm_w;
  float eps;
  const float* cos;               // [m, 64]
  const float* sin;
  const int32_t* rows;
  const int32_t* positions;
  void* q_rot;                    // NULL: plain projection
  void* k_cache;
  void* v_cache;
  int num_rows, max_len;
  const int32_t* block_table;
  int block_size, max_blocks, n_blocks;
  int* err;
};
cudaError_t launch_proj(const ProjArgs& a, cudaStream_t stream);

// Tensor maps (driver entry point resolved at run time; no link-time dependency on libcuda).
bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer);
bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                         uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2);

}  // namespace da
