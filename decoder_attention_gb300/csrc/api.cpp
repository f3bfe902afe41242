// Host side of the C ABI declared in include/decattn.h: argument checks, fp64 RoPE frequency math,
// tensor-map encoding and dispatch to the kernels.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "decattn.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return DA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------------------------------ layer checks

int check_layer(const da_layer* L) {
  if (!L) return fail(DA_ERR_INVALID_ARG, "layer is NULL");
  if (L->dtype != DA_BF16 && L->dtype != DA_FP32) return fail(DA_ERR_INVALID_ARG, "dtype %d is not DA_BF16 or DA_FP32", L->dtype);
  if (L->head_dim != 64 && L->head_dim != 128)
    return fail(DA_ERR_UNSUPPORTED, "head_dim %d is not implemented (64 or 128)", L->head_dim);
  if (L->num_attention_heads < 1 || L->num_key_value_heads < 1)
    return fail(DA_ERR_INVALID_ARG, "head counts must be positive (Hq %d, Hkv %d)", L->num_attention_heads, L->num_key_value_heads);
  if (L->num_attention_heads % L->num_key_value_heads)
    return fail(DA_ERR_INVALID_ARG, "num_attention_heads %d is not a multiple of num_key_value_heads %d",
                L->num_attention_heads, L->num_key_value_heads);
  if (L->rotary_dim < 2 || L->rotary_dim > L->head_dim || (L->rotary_dim & 1))
    return fail(DA_ERR_INVALID_ARG, "rotary_dim %d must be even and in [2, head_dim=%d]", L->rotary_dim, L->head_dim);
  if ((L->q_norm_w == nullptr) != (L->k_norm_w == nullptr))
    return fail(DA_ERR_INVALID_ARG, "q_norm_w and k_norm_w must be both set or both NULL");
  if (!(L->eps >= 0.0) || !std::isfinite(L->eps)) return fail(DA_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (L->window < 0) return fail(DA_ERR_INVALID_ARG, "window %d must be >= 0", L->window);
  if (!(L->softcap >= 0.f) || !std::isfinite(L->softcap)) return fail(DA_ERR_INVALID_ARG, "softcap must be finite and >= 0");
  if (!(L->scale >= 0.f) || !std::isfinite(L->scale)) return fail(DA_ERR_INVALID_ARG, "scale must be finite and >= 0");
  return DA_OK;
}

float layer_scale(const da_layer* L) { return L->scale > 0.f ? L->scale : 1.0f / std::sqrt(static_cast<float>(L->head_dim)); }

// ------------------------------------------------------------------------------------------ frequencies
// Page "42. More models: a registry, scaled RoPE, sliding windows and latent attention", section
// "Scaled RoPE" (rope_inv_freq), and "Model resolution" (Overview) for LongRoPE, restated in fp64.

int compute_freqs(const da_rope_scaling* rs, da::RopeFreqs* f) {
  if (!rs) return fail(DA_ERR_INVALID_ARG, "rope scaling is NULL");
  const int r = rs->rotary_dim;
  if (r < 2 || r > 2 * da::kMaxRotHalf || (r & 1))
    return fail(DA_ERR_INVALID_ARG, "rotary_dim %d must be even and in [2, %d]", r, 2 * da::kMaxRotHalf);
  if (!(rs->theta > 1.0) || !std::isfinite(rs->theta)) return fail(DA_ERR_INVALID_ARG, "rope theta must be finite and > 1");
  const int half = r / 2;
  std::memset(f, 0, sizeof(*f));
  f->half = half;
  f->switch_len = 0x7fffffff;
  f->use_seq_len = 0;
  f->af = 1.0;
  double base[da::kMaxRotHalf];
  for (int i = 0; i < half; ++i) base[i] = 1.0 / std::pow(rs->theta, (2.0 * i) / r);
  const double kPi = 3.14159265358979323846;
  switch (rs->kind) {
    case DA_ROPE_DEFAULT:
      for (int i = 0; i < half; ++i) f->inv_short[i] = base[i];
      break;
    case DA_ROPE_LINEAR:
      if (!(rs->factor > 0.0)) return fail(DA_ERR_INVALID_ARG, "linear rope scaling needs factor > 0");
      for (int i = 0; i < half; ++i) f->inv_short[i] = base[i] / rs->factor;
      break;
    case DA_ROPE_LLAMA3: {
      const double old = rs->original_max_position_embeddings, low = rs->low_freq_factor, high = rs->high_freq_factor;
      if (!(rs->factor > 0.0) || !(old > 0) || !(low > 0.0) || !(high > low))
        return fail(DA_ERR_INVALID_ARG, "llama3 rope scaling needs factor > 0, original > 0, high > low > 0");
      for (int i = 0; i < half; ++i) {
        const double wl = 2.0 * kPi / base[i];
        double v;
        if (wl > old / low) {
          v = base[i] / rs->factor;                           // long wavelengths: interpolated
        } else if (wl >= old / high) {
          const double smooth = (old / wl - low) / (high - low);
          v = (1.0 - smooth) * base[i] / rs->factor + smooth * base[i];
        } else {
          v = base[i];                                        // short wavelengths: kept
        }
        f->inv_short[i] = v;
      }
      break;
    }
    case DA_ROPE_LONGROPE: {
      const int old = rs->original_max_position_embeddings;
      if (!rs->short_factor || !rs->long_factor) return fail(DA_ERR_INVALID_ARG, "longrope needs short_factor and long_factor");
      if (old <= 0) return fail(DA_ERR_INVALID_ARG, "longrope needs original_max_position_embeddings > 0");
      for (int i = 0; i < half; ++i) {
        if (!(rs->short_factor[i] > 0.0) || !(rs->long_factor[i] > 0.0) || !std::isfinite(rs->short_factor[i]) ||
            !std::isfinite(rs->long_factor[i]))
          return fail(DA_ERR_INVALID_ARG, "longrope factors must be finite and > 0 (pair %d)", i);
        f->inv_short[i] = base[i] / rs->short_factor[i];
        f->inv_long[i] = base[i] / rs->long_factor[i];
      }
      f->switch_len = old;
      f->use_seq_len = 1;
      if (rs->attention_factor > 0.0) {
        f->af = rs->attention_factor;
      } else {
        const int mpe = rs->max_position_embeddings > 0 ? rs->max_position_embeddings : old;
        const double s = static_cast<double>(mpe) / old;
        f->af = s <= 1.0 ? 1.0 : std::sqrt(1.0 + std::log(s) / std::log(static_cast<double>(old)));
      }
      break;
    }
    case DA_ROPE_YARN: {
      const double old = rs->original_max_position_embeddings;
      if (!(old > 0)) return fail(DA_ERR_INVALID_ARG, "yarn needs original_max_position_embeddings > 0");
      double factor = rs->factor;
      if (!(factor > 0.0)) {
        if (rs->max_position_embeddings <= 0) return fail(DA_ERR_INVALID_ARG, "yarn needs factor or max_position_embeddings");
        factor = rs->max_position_embeddings / old;
      }
      auto mscale = [](double sc, double m) { return sc <= 1.0 ? 1.0 : 0.1 * m * std::log(sc) + 1.0; };
      if (rs->attention_factor > 0.0)
        f->af = rs->attention_factor;
      else if (rs->mscale > 0.0 && rs->mscale_all_dim > 0.0)
        f->af = mscale(factor, rs->mscale) / mscale(factor, rs->mscale_all_dim);
      else
        f->af = mscale(factor, 1.0);
      // fractional pair index whose wavelength fits `rot` times into the original context
      auto pair_for = [&](double rot) { return r * std::log(old / (rot * 2.0 * kPi)) / (2.0 * std::log(rs->theta)); };
      double lo = pair_for(rs->beta_fast > 0.0 ? rs->beta_fast : 32.0);
      double hi = pair_for(rs->beta_slow > 0.0 ? rs->beta_slow : 1.0);
      if (rs->truncate) {
        lo = std::floor(lo);
        hi = std::ceil(hi);
      }
      lo = std::max(lo, 0.0);
      hi = std::min(hi, static_cast<double>(r - 1));
      const double span = (hi != lo) ? (hi - lo) : 0.001;
      for (int i = 0; i < half; ++i) {
        const double ramp = std::min(1.0, std::max(0.0, (i - lo) / span));   // 0: fast pair, 1: slow pair
        f->inv_short[i] = base[i] / factor * ramp + base[i] * (1.0 - ramp);
      }
      break;
    }
    default:
      return fail(DA_ERR_UNSUPPORTED, "RoPE kind %d is not implemented", rs->kind);
  }
  if (!f->use_seq_len)
    for (int i = 0; i < half; ++i) f->inv_long[i] = f->inv_short[i];
  return DA_OK;
}

// ------------------------------------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

namespace da {

bool encode_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                         uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace da

// ============================================================================================ C ABI

extern "C" {

const char* da_last_error(void) { return g_last_error.c_str(); }

int da_version(void) { return 100; }   // 0.1.0

int da_rope_tables_build(const da_rope_scaling* rs, const int32_t* positions, const int32_t* seq_len, int n,
                         float* cos, float* sin, cudaStream_t stream) {
  da::RopeFreqs f;
  int rc = compute_freqs(rs, &f);
  if (rc) return rc;
  if (n < 0) return fail(DA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (!positions || !cos || !sin) return fail(DA_ERR_INVALID_ARG, "positions, cos and sin must be non-NULL");
  if (f.use_seq_len && !seq_len) return fail(DA_ERR_INVALID_ARG, "longrope needs seq_len per token");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  cudaError_t e = da::launch_rope_tables(f, positions, seq_len, n, cos, sin, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "rope_tables launch");
  return ok();
}

// A paged pool's description, checked; fills the layout fields the kernels read.
static int check_paged(const da_layer* L, const da_paged_kv* kv) {
  if (!kv) return fail(DA_ERR_INVALID_ARG, "the paged pool description is NULL");
  if (!kv->k_pool || !kv->v_pool || !kv->block_table) return fail(DA_ERR_INVALID_ARG, "a pool pointer is NULL");
  if (kv->n_blocks < 1 || kv->block_size < 1 || kv->num_rows < 1 || kv->max_blocks < 1)
    return fail(DA_ERR_INVALID_ARG, "n_blocks, block_size, num_rows and max_blocks must be >= 1");
  if (static_cast<long long>(kv->max_blocks) * kv->block_size > 0x7fffffffLL)
    return fail(DA_ERR_UNSUPPORTED, "max_blocks * block_size exceeds 2^31 positions");
  if (static_cast<long long>(kv->n_blocks) * L->num_key_value_heads * kv->block_size > 0x7fffffffLL)
    return fail(DA_ERR_UNSUPPORTED, "n_blocks * Hkv * block_size exceeds 2^31 key slots");
  if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return fail(DA_ERR_INVALID_ARG, "the pools must be 16-byte aligned");
  return DA_OK;
}

extern "C++" {
template <typename Args>
static void set_paged(Args& a, const da_paged_kv* kv) {
  if (kv) {
    a.block_table = kv->block_table;
    a.block_size = kv->block_size;
    a.max_blocks = kv->max_blocks;
    a.n_blocks = kv->n_blocks;
  } else {
    a.block_table = nullptr;
    a.block_size = a.max_blocks = a.n_blocks = 0;
  }
}
}

// rs != NULL: cos/sin are formed in the kernel from rs, positions and seq_len (cos/sin unused).
static int kv_update_impl(const da_layer* L, const void* q, const void* k, const void* v, int n, const int32_t* rows,
                          const int32_t* positions, const float* cos, const float* sin, void* q_rot, void* k_cache,
                          void* v_cache, int num_rows, int max_len, const da_paged_kv* kv, cudaStream_t stream,
                          const da_rope_scaling* rs = nullptr, const int32_t* seq_len = nullptr) {
  int rc = check_layer(L);
  if (rc) return rc;
  da::RopeFreqs f;
  if (rs) {
    rc = compute_freqs(rs, &f);
    if (rc) return rc;
    if (rs->rotary_dim != L->rotary_dim)
      return fail(DA_ERR_INVALID_ARG, "the scaling's rotary_dim %d differs from the layer's %d", rs->rotary_dim,
                  L->rotary_dim);
    if (!da::kv_update_rope_supported(L->dtype == DA_BF16, L->head_dim, L->rotary_dim))
      return fail(DA_ERR_UNSUPPORTED, "the fused rope form needs bf16, head_dim 128 and rotary_dim a multiple of 16");
  }
  if (n < 0) return fail(DA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (!q || !k || !v || !rows || !positions || (!rs && (!cos || !sin)) || !q_rot || !k_cache || !v_cache)
    return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (rs && f.use_seq_len && !seq_len) return fail(DA_ERR_INVALID_ARG, "longrope needs seq_len per token");
  if (num_rows < 1 || max_len < 1) return fail(DA_ERR_INVALID_ARG, "num_rows and max_len must be >= 1");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (!rs && (!aligned16(cos) || !aligned16(sin))) || !aligned16(L->q_norm_w) || !aligned16(L->k_norm_w))
    return fail(DA_ERR_INVALID_ARG, "q, k, v, q_rot, the caches, cos/sin and the norm weights must be 16-byte aligned");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::KvUpdateArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.n = n;
  a.hq = L->num_attention_heads;
  a.hkv = L->num_key_value_heads;
  a.d = L->head_dim;
  a.rot = L->rotary_dim;
  a.rows = rows;
  a.positions = positions;
  a.cos = cos;
  a.sin = sin;
  a.q_norm_w = L->q_norm_w;
  a.k_norm_w = L->k_norm_w;
  a.eps = static_cast<float>(L->eps);
  a.q_rot = q_rot;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_rows = num_rows;
  a.max_len = max_len;
  set_paged(a, kv);
  a.err = err;
  a.seq_len = seq_len;
  cudaError_t e = rs ? da::launch_kv_update_rope(a, f, stream) : da::launch_kv_update(a, L->dtype == DA_BF16, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kv_cache_update launch");
  return ok();
}

int da_kv_cache_update(const da_layer* L, const void* q, const void* k, const void* v, int n, const int32_t* rows,
                       const int32_t* positions, const float* cos, const float* sin, void* q_rot, void* k_cache,
                       void* v_cache, int num_rows, int max_len, cudaStream_t stream) {
  return kv_update_impl(L, q, k, v, n, rows, positions, cos, sin, q_rot, k_cache, v_cache, num_rows, max_len, nullptr,
                        stream);
}

int da_kv_cache_update_paged(const da_layer* L, const void* q, const void* k, const void* v, int n, const int32_t* rows,
                             const int32_t* positions, const float* cos, const float* sin, void* q_rot,
                             const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return kv_update_impl(L, q, k, v, n, rows, positions, cos, sin, q_rot, kv->k_pool, kv->v_pool, kv->num_rows,
                        kv->max_blocks * kv->block_size, kv, stream);
}

int da_kv_cache_update_rope(const da_layer* L, const da_rope_scaling* rs, const void* q, const void* k, const void* v,
                            int n, const int32_t* rows, const int32_t* positions, const int32_t* seq_len, void* q_rot,
                            void* k_cache, void* v_cache, int num_rows, int max_len, cudaStream_t stream) {
  if (!rs) return fail(DA_ERR_INVALID_ARG, "the rope scaling is NULL");
  return kv_update_impl(L, q, k, v, n, rows, positions, nullptr, nullptr, q_rot, k_cache, v_cache, num_rows, max_len,
                        nullptr, stream, rs, seq_len);
}

int da_kv_cache_update_rope_paged(const da_layer* L, const da_rope_scaling* rs, const void* q, const void* k,
                                  const void* v, int n, const int32_t* rows, const int32_t* positions,
                                  const int32_t* seq_len, void* q_rot, const da_paged_kv* kv, cudaStream_t stream) {
  if (!rs) return fail(DA_ERR_INVALID_ARG, "the rope scaling is NULL");
  int rc = check_layer(L);
  if (rc) return rc;
  if (n == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return kv_update_impl(L, q, k, v, n, rows, positions, nullptr, nullptr, q_rot, kv->k_pool, kv->v_pool, kv->num_rows,
                        kv->max_blocks * kv->block_size, kv, stream, rs, seq_len);
}

static int attn_common_checks(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache,
                              int num_rows, int max_len, int n_seqs, const int32_t* rows, void* out,
                              bool paged = false) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_seqs < 0) return fail(DA_ERR_INVALID_ARG, "n_seqs = %d < 0", n_seqs);
  if (n_seqs > 65535) return fail(DA_ERR_UNSUPPORTED, "n_seqs = %d > 65535 per call", n_seqs);
  if (n_seqs == 0) return DA_OK;
  if (!q_rot || !k_cache || !v_cache || !rows || !out) return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_rows < 1 || max_len < 1) return fail(DA_ERR_INVALID_ARG, "num_rows and max_len must be >= 1");
  if (!paged && static_cast<long long>(num_rows) * L->num_key_value_heads * max_len > 0x7fffffffLL)
    return fail(DA_ERR_UNSUPPORTED, "num_rows * Hkv * max_len exceeds 2^31 key slots");
  if (!aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(DA_ERR_INVALID_ARG, "q_rot, the caches and out must be 16-byte aligned");
  return DA_OK;
}

static da::AttnArgs make_args(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache,
                              int num_rows, int max_len, int n_seqs, const int32_t* rows, const int32_t* key_positions,
                              void* out, int* err) {
  da::AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q_rot = q_rot;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.out = out;
  a.hq = L->num_attention_heads;
  a.hkv = L->num_key_value_heads;
  a.d = L->head_dim;
  a.num_rows = num_rows;
  a.max_len = max_len;
  a.n_seqs = n_seqs;
  a.rows = rows;
  a.key_positions = key_positions;
  a.window = L->window;
  a.softcap = L->softcap;
  a.scale = layer_scale(L);
  a.sinks = L->sinks;
  a.err = err;
  return a;
}

// check_only: every host check, then return without enqueueing. max_ctas: cap on the tcgen05 prefill's
// persistent grid (0: one CTA per SM).
static int prefill_impl(const da_layer* L, const void* q_rot, int n_tokens, const void* k_cache, const void* v_cache,
                        int num_rows, int max_len, int n_seqs, const int32_t* q_start, const int32_t* rows,
                        const int32_t* first_pos, int max_q_len, const int32_t* key_positions, void* out,
                        const da_paged_kv* kv, cudaStream_t stream, bool check_only = false, int max_ctas = 0) {
  int rc = attn_common_checks(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, out, kv != nullptr);
  if (rc) return rc;
  if (n_tokens < 0 || max_q_len < 0) return fail(DA_ERR_INVALID_ARG, "n_tokens and max_q_len must be >= 0");
  if (n_seqs == 0 || n_tokens == 0 || max_q_len == 0) return ok();
  if (!q_start || !first_pos) return fail(DA_ERR_INVALID_ARG, "q_start and first_pos must be non-NULL");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::AttnArgs a = make_args(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, key_positions, out, err);
  a.q_start = q_start;
  a.first_pos = first_pos;
  a.max_q_len = max_q_len;
  a.n_tokens = n_tokens;
  set_paged(a, kv);
  a.max_ctas = max_ctas;
  const bool fast = L->dtype == DA_BF16 && L->head_dim == 128 && key_positions == nullptr &&
                    (kv == nullptr || kv->block_size % 64 == 0);
  if (check_only) return ok();
  cudaError_t e = fast ? da::launch_prefill_bf16(a, stream) : da::launch_attn_generic(a, L->dtype == DA_BF16, stream);
  if (e != cudaSuccess) return cuda_fail(e, fast ? "prefill (tcgen05) launch" : "prefill (generic) launch");
  return ok();
}

int da_attn_prefill(const da_layer* L, const void* q_rot, int n_tokens, const void* k_cache, const void* v_cache,
                    int num_rows, int max_len, int n_seqs, const int32_t* q_start, const int32_t* rows,
                    const int32_t* first_pos, int max_q_len, const int32_t* key_positions, void* out, void* workspace,
                    size_t ws_bytes, cudaStream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  return prefill_impl(L, q_rot, n_tokens, k_cache, v_cache, num_rows, max_len, n_seqs, q_start, rows, first_pos,
                      max_q_len, key_positions, out, nullptr, stream);
}

int da_attn_prefill_paged(const da_layer* L, const void* q_rot, int n_tokens, const da_paged_kv* kv, int n_seqs,
                          const int32_t* q_start, const int32_t* rows, const int32_t* first_pos, int max_q_len,
                          void* out, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_seqs == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return prefill_impl(L, q_rot, n_tokens, kv->k_pool, kv->v_pool, kv->num_rows, kv->max_blocks * kv->block_size,
                      n_seqs, q_start, rows, first_pos, max_q_len, nullptr, out, kv, stream);
}

static bool decode_fast(const da_layer* L, const int32_t* key_positions) {
  return L->dtype == DA_BF16 && L->head_dim == 128 && key_positions == nullptr &&
         L->num_attention_heads / L->num_key_value_heads <= 8;
}

size_t da_decode_workspace_bytes(const da_layer* L, int n_seqs, int max_len) {
  if (check_layer(L) != DA_OK || n_seqs <= 0 || max_len <= 0) return 0;
  if (!decode_fast(L, nullptr)) return 0;
  const da::DecodePlan p = da::decode_plan(L->num_key_value_heads, n_seqs, max_len, L->window, false);
  return da::decode_workspace_bytes(L->num_attention_heads, n_seqs, p);
}

size_t da_decode_workspace_bytes_paged(const da_layer* L, int n_seqs, int max_positions) {
  if (check_layer(L) != DA_OK || n_seqs <= 0 || max_positions <= 0) return 0;
  if (!decode_fast(L, nullptr)) return 0;
  // chunks start at the window start rounded down to a 64-key tile: up to 63 more keys per sequence
  const da::DecodePlan p = da::decode_plan(L->num_key_value_heads, n_seqs, max_positions, L->window, true);
  return da::decode_workspace_bytes(L->num_attention_heads, n_seqs, p);
}

static int decode_impl(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache, int num_rows,
                       int max_len, int n_seqs, const int32_t* rows, const int32_t* positions,
                       const int32_t* key_positions, void* out, void* workspace, size_t ws_bytes,
                       const da_paged_kv* kv, cudaStream_t stream, bool check_only = false) {
  int rc = attn_common_checks(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, out, kv != nullptr);
  if (rc) return rc;
  if (n_seqs == 0) return ok();
  if (!positions) return fail(DA_ERR_INVALID_ARG, "positions must be non-NULL");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::AttnArgs a = make_args(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, key_positions, out, err);
  a.positions = positions;
  a.max_q_len = 1;
  a.n_tokens = n_seqs;
  set_paged(a, kv);
  if (!decode_fast(L, key_positions) || (kv && kv->block_size % 64 != 0)) {
    if (check_only) return ok();
    cudaError_t e = da::launch_attn_generic(a, L->dtype == DA_BF16, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode (generic) launch");
    return ok();
  }
  const da::DecodePlan p = da::decode_plan(L->num_key_value_heads, n_seqs, max_len, L->window, kv != nullptr);
  const size_t need = da::decode_workspace_bytes(L->num_attention_heads, n_seqs, p);
  if (!workspace || ws_bytes < need)
    return fail(DA_ERR_INVALID_ARG, "decode workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
  if (!aligned16(workspace)) return fail(DA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (check_only) return ok();
  cudaError_t e = da::launch_decode_bf16(a, p, workspace, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode (split-K) launch");
  return ok();
}

int da_attn_decode(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache, int num_rows,
                   int max_len, int n_seqs, const int32_t* rows, const int32_t* positions,
                   const int32_t* key_positions, void* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  return decode_impl(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, positions, key_positions, out,
                     workspace, ws_bytes, nullptr, stream);
}

int da_attn_decode_paged(const da_layer* L, const void* q_rot, const da_paged_kv* kv, int n_seqs, const int32_t* rows,
                         const int32_t* positions, void* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_seqs == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return decode_impl(L, q_rot, kv->k_pool, kv->v_pool, kv->num_rows, kv->max_blocks * kv->block_size, n_seqs, rows,
                     positions, nullptr, out, workspace, ws_bytes, kv, stream);
}

// ------------------------------------------------------------------------------------------ mixed batches

namespace {

// The stream a mixed call forks onto and its fork/join events: one set per device, created on first use and
// kept until the process exits. g_side_mu is held while a call enqueues, so that no other call records the
// shared events between another's record and wait.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

// Rates of the two kernels on GB300 that the split below models (measured: the tcgen05 prefill at 1092
// TFLOP/s over 152 SMs on contiguous caches, about 0.8 of that over a paged pool; the split-K decode at 7.2
// TB/s on the whole GPU, ~100 GB/s per SM or more when it has a few dozen SMs to itself).
constexpr double kPrefillFlopsPerSm = 7.2e12;
constexpr double kPagedPrefillRate = 0.8;
constexpr double kDecodeBytesPerSm = 1.0e11;
constexpr double kDecodeBytesAll = 7.2e12;

// Persistent prefill CTAs for a prefill and a decode that share the GPU; n_sm means one after the other.
// With P prefill CTAs (one per SM: nothing else fits beside one) the decode's blocks get the other SMs, and
// once the prefill ends they spread over all of them (the persistent prefill cannot grow into SMs that the
// decode leaves). P minimises the modelled end of both, and is used only when that beats running them in turn
// by more than 3% (the fork and join, and the model's own error, cost a few).
int mixed_prefill_ctas(int n_sm, double flops, double bytes, bool paged) {
  const double rate = kPrefillFlopsPerSm * (paged ? kPagedPrefillRate : 1.0);
  const double serial = flops / (n_sm * rate) + bytes / kDecodeBytesAll;
  double best = serial;
  int best_p = n_sm;
  for (int p = std::max(1, n_sm / 4); p < n_sm; ++p) {
    const double t_pf = flops / (p * rate);
    const double bw = std::min((n_sm - p) * kDecodeBytesPerSm, kDecodeBytesAll);
    const double t = bytes <= t_pf * bw ? t_pf : t_pf + (bytes - t_pf * bw) / kDecodeBytesAll;
    if (t < best) {
      best = t;
      best_p = p;
    }
  }
  return best < 0.97 * serial ? best_p : n_sm;
}

}  // namespace

// The split for a layer's hints: prefill FLOPs 4 d Hq pairs, decode bytes keys * 2 Hkv d * 2 (bf16).
static int mixed_split(const da_layer* L, int n_sm, double prefill_pairs, double decode_keys, bool paged) {
  const double flops = 4.0 * L->head_dim * L->num_attention_heads * prefill_pairs;
  const double bytes = decode_keys * 2.0 * L->num_key_value_heads * L->head_dim * 2.0;
  return mixed_prefill_ctas(n_sm, flops, bytes, paged);
}

int da_attn_mixed_prefill_sms(const da_layer* L, int n_sm, double prefill_pairs, double decode_keys) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_sm < 1) return fail(DA_ERR_INVALID_ARG, "n_sm = %d < 1", n_sm);
  if (!(prefill_pairs >= 0.0) || !(decode_keys >= 0.0) || !std::isfinite(prefill_pairs) ||
      !std::isfinite(decode_keys))
    return fail(DA_ERR_INVALID_ARG, "prefill_pairs and decode_keys must be finite and >= 0");
  ok();
  if (prefill_pairs == 0.0 || decode_keys == 0.0) return n_sm;
  return mixed_split(L, n_sm, prefill_pairs, decode_keys, false);
}

static int mixed_impl(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache, int num_rows,
                      int max_len, int n_tokens, int n_seqs, const int32_t* q_start, const int32_t* chunk_rows,
                      const int32_t* first_pos, int max_q_len, int n_decode, const int32_t* dec_rows,
                      const int32_t* dec_positions, double prefill_pairs, double decode_keys, void* out,
                      void* workspace, size_t ws_bytes, const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_tokens < 0 || n_decode < 0) return fail(DA_ERR_INVALID_ARG, "n_tokens and n_decode must be >= 0");
  if (!(prefill_pairs >= 0.0) || !(decode_keys >= 0.0) || !std::isfinite(prefill_pairs) ||
      !std::isfinite(decode_keys))
    return fail(DA_ERR_INVALID_ARG, "prefill_pairs and decode_keys must be finite and >= 0");
  // decode tokens follow the chunks' tokens in q_rot and out
  const size_t row_bytes =
      static_cast<size_t>(L->num_attention_heads) * L->head_dim * (L->dtype == DA_BF16 ? 2 : 4);
  const void* q_dec = q_rot ? static_cast<const uint8_t*>(q_rot) + static_cast<size_t>(n_tokens) * row_bytes : nullptr;
  void* out_dec = out ? static_cast<uint8_t*>(out) + static_cast<size_t>(n_tokens) * row_bytes : nullptr;
  auto prefill = [&](cudaStream_t st, bool check_only, int max_ctas) {
    return prefill_impl(L, q_rot, n_tokens, k_cache, v_cache, num_rows, max_len, n_seqs, q_start, chunk_rows,
                        first_pos, max_q_len, nullptr, out, kv, st, check_only, max_ctas);
  };
  auto decode = [&](cudaStream_t st, bool check_only) {
    return decode_impl(L, q_dec, k_cache, v_cache, num_rows, max_len, n_decode, dec_rows, dec_positions, nullptr,
                       out_dec, workspace, ws_bytes, kv, st, check_only);
  };
  // every check of both parts before anything is enqueued
  rc = prefill(stream, true, 0);
  if (rc) return rc;
  rc = decode(stream, true);
  if (rc) return rc;

  const bool pf_work = n_seqs > 0 && n_tokens > 0 && max_q_len > 0, dec_work = n_decode > 0;
  const bool tc = L->dtype == DA_BF16 && L->head_dim == 128 && L->num_attention_heads / L->num_key_value_heads <= 8 &&
                  (kv == nullptr || kv->block_size % 64 == 0);
  int dev = 0, n_sm = 0, p = 0;
  if (pf_work && dec_work && tc && prefill_pairs > 0.0 && decode_keys > 0.0) {
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    p = mixed_split(L, n_sm, prefill_pairs, decode_keys, kv != nullptr);
  }
  if (p == 0 || p >= n_sm || dev >= kMaxDevices) {   // one after the other on `stream`
    rc = prefill(stream, false, 0);
    if (rc) return rc;
    return decode(stream, false);
  }

  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    cudaError_t e = cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (ss.join) cudaEventDestroy(ss.join);
      if (ss.fork) cudaEventDestroy(ss.fork);
      if (ss.stream) cudaStreamDestroy(ss.stream);
      ss = SideStream{};
      return cuda_fail(e, "mixed batch: side stream");
    }
  }
  cudaError_t e = cudaEventRecord(ss.fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ss.stream, ss.fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "mixed batch: fork");
  // the prefill first, so that its persistent CTAs take their SMs before the decode's blocks fill the rest
  rc = prefill(stream, false, p);
  const int rc_dec = rc ? rc : decode(ss.stream, false);
  e = cudaEventRecord(ss.join, ss.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ss.join, 0);
  if (rc || rc_dec) return rc ? rc : rc_dec;
  if (e != cudaSuccess) return cuda_fail(e, "mixed batch: join");
  return ok();
}

int da_attn_mixed(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache, int num_rows,
                  int max_len, int n_tokens, int n_seqs, const int32_t* q_start, const int32_t* chunk_rows,
                  const int32_t* first_pos, int max_q_len, int n_decode, const int32_t* dec_rows,
                  const int32_t* dec_positions, double prefill_pairs, double decode_keys, void* out, void* workspace,
                  size_t ws_bytes, cudaStream_t stream) {
  return mixed_impl(L, q_rot, k_cache, v_cache, num_rows, max_len, n_tokens, n_seqs, q_start, chunk_rows, first_pos,
                    max_q_len, n_decode, dec_rows, dec_positions, prefill_pairs, decode_keys, out, workspace, ws_bytes,
                    nullptr, stream);
}

int da_attn_mixed_paged(const da_layer* L, const void* q_rot, const da_paged_kv* kv, int n_tokens, int n_seqs,
                        const int32_t* q_start, const int32_t* chunk_rows, const int32_t* first_pos, int max_q_len,
                        int n_decode, const int32_t* dec_rows, const int32_t* dec_positions, double prefill_pairs,
                        double decode_keys, void* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n_seqs == 0 && n_decode == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return mixed_impl(L, q_rot, kv->k_pool, kv->v_pool, kv->num_rows, kv->max_blocks * kv->block_size, n_tokens, n_seqs,
                    q_start, chunk_rows, first_pos, max_q_len, n_decode, dec_rows, dec_positions, prefill_pairs,
                    decode_keys, out, workspace, ws_bytes, kv, stream);
}

int da_attn_decode_noalloc(const da_layer* L, const void* q_rot, const void* k_cache, const void* v_cache,
                           int num_rows, int max_len, int n_seqs, const int32_t* rows, const int32_t* positions,
                           const int32_t* key_positions, void* out, cudaStream_t stream) {
  int rc = attn_common_checks(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, out);
  if (rc) return rc;
  if (n_seqs == 0) return ok();
  if (!positions) return fail(DA_ERR_INVALID_ARG, "positions must be non-NULL");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::AttnArgs a = make_args(L, q_rot, k_cache, v_cache, num_rows, max_len, n_seqs, rows, key_positions, out, err);
  a.positions = positions;
  a.max_q_len = 1;
  a.n_tokens = n_seqs;
  if (!decode_fast(L, key_positions)) {   // the CUDA-core kernel needs no scratch
    cudaError_t e = da::launch_attn_generic(a, L->dtype == DA_BF16, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode (generic) launch");
    return ok();
  }
  const da::DecodePlan p = da::decode_plan(L->num_key_value_heads, n_seqs, max_len, L->window, false);
  const size_t need = da::decode_workspace_bytes(L->num_attention_heads, n_seqs, p);
  if (need > da::kDecodeStaticScratchBytes)
    return fail(DA_ERR_INVALID_ARG,
                "decode needs %zu bytes of scratch, more than the %zu bytes of the library's fixed scratch; "
                "use da_attn_decode with a caller-provided workspace or split the batch",
                need, da::kDecodeStaticScratchBytes);
  void* scratch = da::static_scratch();
  if (!scratch) return fail(DA_ERR_CUDA, "cannot locate the fixed decode scratch on this device");
  cudaError_t e = da::launch_decode_bf16(a, p, scratch, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode (split-K, fixed scratch) launch");
  return ok();
}

size_t da_decode_noalloc_max_scratch_bytes(void) { return da::kDecodeStaticScratchBytes; }

int da_check_device_error(cudaStream_t stream) {
  int flags = 0;
  if (da::read_and_clear_error_word(stream, &flags) != DA_OK)
    return fail(DA_ERR_CUDA, "could not read the device error word: %s", cudaGetErrorString(cudaGetLastError()));
  if (flags & da::kErrTimeout) return fail(DA_ERR_TIMEOUT, "a kernel gave up a bounded wait (timeout)");
  if (flags & da::kErrIndex) return fail(DA_ERR_DEVICE_INDEX, "a kernel met a row, position or slot out of range");
  return ok();
}

// ---------------------------------------------------------------------------------------------- MLA

static int check_mla_layer(const da_mla_layer* L) {
  if (!L) return fail(DA_ERR_INVALID_ARG, "layer is NULL");
  if (L->kv_lora_rank != 512 || L->qk_rope_dim != 64)
    return fail(DA_ERR_UNSUPPORTED, "MLA supports kv_lora_rank 512 and qk_rope_dim 64 (got %d, %d)", L->kv_lora_rank,
                L->qk_rope_dim);
  if (L->num_heads < 8 || L->num_heads % 8 != 0 || L->num_heads > 4096)
    return fail(DA_ERR_UNSUPPORTED, "MLA num_heads must be a positive multiple of 8 (got %d)", L->num_heads);
  if (!(L->scale > 0.f) || !std::isfinite(L->scale)) return fail(DA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (L->window < 0) return fail(DA_ERR_INVALID_ARG, "window = %d < 0", L->window);
  return DA_OK;
}

static int mla_update_impl(const da_mla_layer* L, const void* latent, const void* k_rope, int n, const int32_t* rows,
                           const int32_t* positions, const float* cos, const float* sin, void* q, void* cache,
                           int num_rows, int max_len, const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_mla_layer(L);
  if (rc) return rc;
  if (n < 0) return fail(DA_ERR_INVALID_ARG, "n = %d < 0", n);
  if (n == 0) return ok();
  if (!latent || !k_rope || !rows || !positions || !cos || !sin || !cache)
    return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_rows < 1 || max_len < 1) return fail(DA_ERR_INVALID_ARG, "num_rows and max_len must be >= 1");
  if (!aligned16(latent) || !aligned16(cache) || !aligned16(q) || (reinterpret_cast<uintptr_t>(k_rope) & 3))
    return fail(DA_ERR_INVALID_ARG, "latent, q and the cache must be 16-byte aligned, k_rope 4-byte aligned");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::MlaUpdateArgs a;
  std::memset(&a, 0, sizeof(a));
  a.latent = latent;
  a.k_rope = k_rope;
  a.rows = rows;
  a.positions = positions;
  a.cos = cos;
  a.sin = sin;
  a.q = q;
  a.cache = cache;
  a.n = n;
  a.hq = L->num_heads;
  a.num_rows = num_rows;
  a.max_len = max_len;
  set_paged(a, kv);
  a.err = err;
  cudaError_t e = da::launch_mla_update(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "MLA cache update launch");
  return ok();
}

int da_mla_cache_update(const da_mla_layer* L, const void* latent, const void* k_rope, int n, const int32_t* rows,
                        const int32_t* positions, const float* cos, const float* sin, void* q, void* cache,
                        int num_rows, int max_len, cudaStream_t stream) {
  return mla_update_impl(L, latent, k_rope, n, rows, positions, cos, sin, q, cache, num_rows, max_len, nullptr,
                         stream);
}

static int check_mla_paged(const da_mla_layer* L, const da_paged_kv* kv) {
  if (!kv) return fail(DA_ERR_INVALID_ARG, "the paged pool description is NULL");
  if (!kv->k_pool || !kv->block_table) return fail(DA_ERR_INVALID_ARG, "a pool pointer is NULL");
  if (kv->n_blocks < 1 || kv->block_size < 1 || kv->num_rows < 1 || kv->max_blocks < 1)
    return fail(DA_ERR_INVALID_ARG, "n_blocks, block_size, num_rows and max_blocks must be >= 1");
  if (static_cast<long long>(kv->max_blocks) * kv->block_size > 0x7fffffffLL ||
      static_cast<long long>(kv->n_blocks) * kv->block_size > 0x7fffffffLL)
    return fail(DA_ERR_UNSUPPORTED, "the pool or a row exceeds 2^31 positions");
  if (!aligned16(kv->k_pool)) return fail(DA_ERR_INVALID_ARG, "the pool must be 16-byte aligned");
  (void)L;
  return DA_OK;
}

int da_mla_cache_update_paged(const da_mla_layer* L, const void* latent, const void* k_rope, int n,
                              const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                              void* q, const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_mla_layer(L);
  if (rc) return rc;
  if (n == 0) return ok();
  rc = check_mla_paged(L, kv);
  if (rc) return rc;
  return mla_update_impl(L, latent, k_rope, n, rows, positions, cos, sin, q, kv->k_pool, kv->num_rows,
                         kv->max_blocks * kv->block_size, kv, stream);
}

double da_mla_softmax_scale(int qk_nope_head_dim, int qk_rope_head_dim, double factor, double mscale_all_dim) {
  if (qk_nope_head_dim < 0 || qk_rope_head_dim < 0 || qk_nope_head_dim + qk_rope_head_dim <= 0)
    return std::nan("");
  double scale = 1.0 / std::sqrt(static_cast<double>(qk_nope_head_dim + qk_rope_head_dim));
  if (mscale_all_dim > 0.0 && factor > 1.0) {
    const double m = 0.1 * mscale_all_dim * std::log(factor) + 1.0;
    scale *= m * m;
  }
  return scale;
}

size_t da_mla_workspace_bytes(const da_mla_layer* L, int n_seqs, int max_len) {
  if (check_mla_layer(L) != DA_OK || n_seqs <= 0 || max_len <= 0) return 0;
  return da::mla_workspace_bytes(L->num_heads, n_seqs, da::mla_plan(L->num_heads, n_seqs, max_len, L->window, false));
}

size_t da_mla_workspace_bytes_paged(const da_mla_layer* L, int n_seqs, int max_positions) {
  if (check_mla_layer(L) != DA_OK || n_seqs <= 0 || max_positions <= 0) return 0;
  return da::mla_workspace_bytes(L->num_heads, n_seqs,
                                 da::mla_plan(L->num_heads, n_seqs, max_positions, L->window, true));
}

static int mla_decode_impl(const da_mla_layer* L, const void* q, const void* cache, int num_rows, int max_len,
                           int n_seqs, const int32_t* rows, const int32_t* positions, void* out, void* workspace,
                           size_t ws_bytes, const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_mla_layer(L);
  if (rc) return rc;
  if (n_seqs < 0) return fail(DA_ERR_INVALID_ARG, "n_seqs = %d < 0", n_seqs);
  if (n_seqs > 65535) return fail(DA_ERR_UNSUPPORTED, "n_seqs = %d > 65535 per call", n_seqs);
  if (n_seqs == 0) return ok();
  if (!q || !cache || !rows || !positions || !out) return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_rows < 1 || max_len < 1) return fail(DA_ERR_INVALID_ARG, "num_rows and max_len must be >= 1");
  if (!kv && static_cast<long long>(num_rows) * max_len > 0x7fffffffLL)
    return fail(DA_ERR_UNSUPPORTED, "num_rows * max_len exceeds 2^31 rows");
  if (kv && kv->block_size % 64 != 0)
    return fail(DA_ERR_UNSUPPORTED, "MLA decode over a pool needs a block size that is a multiple of 64");
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out))
    return fail(DA_ERR_INVALID_ARG, "q, the cache and out must be 16-byte aligned");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  const da::MlaPlan p = da::mla_plan(L->num_heads, n_seqs, max_len, L->window, kv != nullptr);
  const size_t need = da::mla_workspace_bytes(L->num_heads, n_seqs, p);
  if (!workspace || ws_bytes < need)
    return fail(DA_ERR_INVALID_ARG, "MLA workspace of %zu bytes is smaller than the %zu needed", ws_bytes, need);
  if (!aligned16(workspace)) return fail(DA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  da::MlaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = q;
  a.cache = cache;
  a.out = out;
  a.hq = L->num_heads;
  a.num_rows = num_rows;
  a.max_len = max_len;
  a.n_seqs = n_seqs;
  a.window = L->window;
  a.scale = L->scale;
  a.rows = rows;
  a.positions = positions;
  set_paged(a, kv);
  a.err = err;
  cudaError_t e = da::launch_mla_decode(a, p, workspace, stream);
  if (e != cudaSuccess) return cuda_fail(e, "MLA decode launch");
  return ok();
}

int da_mla_decode(const da_mla_layer* L, const void* q, const void* cache, int num_rows, int max_len, int n_seqs,
                  const int32_t* rows, const int32_t* positions, void* out, void* workspace, size_t ws_bytes,
                  cudaStream_t stream) {
  return mla_decode_impl(L, q, cache, num_rows, max_len, n_seqs, rows, positions, out, workspace, ws_bytes, nullptr,
                         stream);
}

int da_mla_decode_paged(const da_mla_layer* L, const void* q, const da_paged_kv* kv, int n_seqs, const int32_t* rows,
                        const int32_t* positions, void* out, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_mla_layer(L);
  if (rc) return rc;
  if (n_seqs == 0) return ok();
  rc = check_mla_paged(L, kv);
  if (rc) return rc;
  return mla_decode_impl(L, q, kv->k_pool, kv->num_rows, kv->max_blocks * kv->block_size, n_seqs, rows, positions,
                         out, workspace, ws_bytes, kv, stream);
}

// ---------------------------------------------------------------------------------------------- projections

static int qkv_proj_impl(const da_layer* L, const void* x, const void* w, const float* bias, int n, int hidden,
                         const int32_t* rows, const int32_t* positions, const float* cos, const float* sin, void* q_rot,
                         void* k_cache, void* v_cache, int num_rows, int max_len, const da_paged_kv* kv,
                         cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n < 0 || hidden < 0) return fail(DA_ERR_INVALID_ARG, "n and hidden must be >= 0");
  if (n == 0) return ok();
  if (L->dtype != DA_BF16 || L->head_dim != 128 || L->rotary_dim != 128)
    return fail(DA_ERR_UNSUPPORTED, "the fused projection needs bf16, head_dim 128 and all 128 dims rotated");
  const int heads = L->num_attention_heads + 2 * L->num_key_value_heads;
  if (heads % 2 != 0) return fail(DA_ERR_UNSUPPORTED, "Hq + 2 Hkv must be even (256-wide output tiles)");
  if (hidden < 64 || hidden % 64 != 0) return fail(DA_ERR_UNSUPPORTED, "hidden must be a positive multiple of 64");
  if (!x || !w || !rows || !positions || !cos || !sin || !q_rot || !k_cache || !v_cache)
    return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (num_rows < 1 || max_len < 1) return fail(DA_ERR_INVALID_ARG, "num_rows and max_len must be >= 1");
  if (!aligned16(x) || !aligned16(w) || !aligned16(q_rot) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(bias) || !aligned16(cos) || !aligned16(sin) || !aligned16(L->q_norm_w) || !aligned16(L->k_norm_w))
    return fail(DA_ERR_INVALID_ARG, "x, w, q_rot, the caches, bias, cos/sin and the norm weights must be 16-byte aligned");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::ProjArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.w = w;
  a.bias = bias;
  a.m = n;
  a.n = heads * 128;
  a.k = hidden;
  a.hq = L->num_attention_heads;
  a.hkv = L->num_key_value_heads;
  a.q_norm_w = L->q_norm_w;
  a.k_norm_w = L->k_norm_w;
  a.eps = static_cast<float>(L->eps);
  a.cos = cos;
  a.sin = sin;
  a.rows = rows;
  a.positions = positions;
  a.q_rot = q_rot;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_rows = num_rows;
  a.max_len = max_len;
  set_paged(a, kv);
  a.err = err;
  cudaError_t e = da::launch_proj(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fused QKV projection launch");
  return ok();
}

int da_qkv_project_update(const da_layer* L, const void* x, const void* w_qkv, const float* bias, int n, int hidden,
                          const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                          void* q_rot, void* k_cache, void* v_cache, int num_rows, int max_len, cudaStream_t stream) {
  return qkv_proj_impl(L, x, w_qkv, bias, n, hidden, rows, positions, cos, sin, q_rot, k_cache, v_cache, num_rows,
                       max_len, nullptr, stream);
}

int da_qkv_project_update_paged(const da_layer* L, const void* x, const void* w_qkv, const float* bias, int n,
                                int hidden, const int32_t* rows, const int32_t* positions, const float* cos,
                                const float* sin, void* q_rot, const da_paged_kv* kv, cudaStream_t stream) {
  int rc = check_layer(L);
  if (rc) return rc;
  if (n == 0) return ok();
  rc = check_paged(L, kv);
  if (rc) return rc;
  return qkv_proj_impl(L, x, w_qkv, bias, n, hidden, rows, positions, cos, sin, q_rot, kv->k_pool, kv->v_pool,
                       kv->num_rows, kv->max_blocks * kv->block_size, kv, stream);
}

int da_linear(const void* x, const void* w, const float* bias, int m, int n, int k, void* y, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return fail(DA_ERR_INVALID_ARG, "m, n and k must be >= 0");
  if (m == 0) return ok();
  if (n < 256 || n % 256 != 0) return fail(DA_ERR_UNSUPPORTED, "n must be a positive multiple of 256");
  if (k < 64 || k % 64 != 0) return fail(DA_ERR_UNSUPPORTED, "k must be a positive multiple of 64");
  if (!x || !w || !y) return fail(DA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(bias))
    return fail(DA_ERR_INVALID_ARG, "x, w, y and bias must be 16-byte aligned");
  int* err = da::error_word_ptr();
  if (!err) return fail(DA_ERR_CUDA, "cannot locate the device error word (no CUDA device?)");
  da::ProjArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.w = w;
  a.bias = bias;
  a.m = m;
  a.n = n;
  a.k = k;
  a.y = y;
  a.err = err;
  cudaError_t e = da::launch_proj(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "linear (tcgen05 GEMM) launch");
  return ok();
}

}  // extern "C"
