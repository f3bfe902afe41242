/*
 * decattn.h -- C ABI of the GB300 (sm_103a) attention step of a rotary, grouped-query decoder layer.
 *
 * The step is the part of DecoderAttention.forward between the q/k/v projections and o_proj, as the page
 * "42. More models: a registry, scaled RoPE, sliding windows and latent attention" (section "What differs
 * between model families") writes it:
 *
 *     q, k = q_norm(q), k_norm(k)            (optional per-head RMSNorm; Qwen3)
 *     q, k = apply_rope(q, cos, sin), ...    (RoPE with the model's frequency scaling)
 *     k, v, key_positions = cache.update(layer, k, v, positions, rows)
 *     allowed = window_mask(qp, kp, sliding_window)          (only on windowed layers)
 *     y = causal_attention(q, k, v, positions, key_positions, allowed)
 *
 * Four calls carry it: da_rope_tables_build (cos/sin per token), da_kv_cache_update (norm + RoPE + cache
 * write), da_attn_prefill and da_attn_decode (attention over the cache).
 *
 * Conventions shared by every call:
 *  - Pointers marked "device" are CUDA device (or managed) memory; "host" pointers are read during the call
 *    only. The caller owns every buffer; the library allocates no memory and frees none.
 *  - Every call is asynchronous on `stream` and returns after enqueueing. Arguments that can be checked on the
 *    host are checked before anything is enqueued; a failed check returns a negative code, enqueues nothing
 *    and leaves a message for da_last_error(). Index violations found on the device (a row, position or
 *    slot out of range) skip the offending access and set a device error word, which da_check_device_error
 *    reports.
 *  - Tensor layouts are dense and row-major (last index fastest):
 *      q, q_rot, out      [N, Hq, d]      one row per token
 *      k, v               [N, Hkv, d]
 *      k_cache, v_cache   [R, Hkv, M, d]  R cache rows (sequences), M positions per row; the slot of a
 *                                          key is its position (slot index = position)
 *      cos, sin           [N, r/2] fp32   r = rotary_dim
 *    Element type: bf16 (DA_BF16) or fp32 (DA_FP32) for q/k/v/caches/out, as da_layer.dtype says.
 *  - Window: w = da_layer.window; 0 means full attention. A key at position j is visible to a query at
 *    position p iff j <= p and, when w > 0, p - j <= w - 1 (page 1, "Sliding windows": keys more than w - 1
 *    positions back are masked).
 *  - GQA: query head h reads KV head floor(h / (Hq / Hkv)).
 */
#ifndef DECATTN_H
#define DECATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define DA_OK                 0
#define DA_ERR_INVALID_ARG   (-1)   /* a host-checkable argument is out of range or inconsistent   */
#define DA_ERR_UNSUPPORTED   (-2)   /* a valid configuration this library does not implement      */
#define DA_ERR_CUDA          (-3)   /* a CUDA runtime call failed (message names it)              */
#define DA_ERR_DEVICE_INDEX  (-4)   /* da_check_device_error: a kernel met an out-of-range index   */
#define DA_ERR_TIMEOUT       (-5)   /* da_check_device_error: a kernel gave up a bounded wait      */
#define DA_ERR_OUT_OF_BLOCKS (-6)   /* da_block_pool_reserve: not enough free blocks (nothing done) */

/* RoPE frequency scaling kinds (page 1, "Scaled RoPE", rope_inv_freq; "Model resolution", Overview,
 * for longrope). */
typedef enum {
    DA_ROPE_DEFAULT  = 0,   /* base_i = theta^(-2i/r)                                              */
    DA_ROPE_LINEAR   = 1,   /* base / factor                                                       */
    DA_ROPE_LLAMA3   = 2,   /* keep short wavelengths, divide long ones by factor, blend between   */
    DA_ROPE_LONGROPE = 3,   /* base / short_factor_i, or base / long_factor_i past the original    */
                            /* context; cos and sin times the attention factor                     */
    DA_ROPE_YARN     = 4    /* ramp between beta_fast/beta_slow pairs; attention factor (mscale)   */
} da_rope_kind;

typedef enum { DA_BF16 = 0, DA_FP32 = 1 } da_dtype;

/* The rope_scaling dict of config.json plus rope_theta and the rotated width. */
typedef struct {
    int    kind;                              /* da_rope_kind                                        */
    double theta;                             /* rope_theta (> 1)                                    */
    int    rotary_dim;                        /* r: even, 2 <= r <= 256 (d * partial_rotary_factor) */
    double factor;                            /* linear, llama3, yarn (yarn: <= 0 means            */
                                              /*   max_position_embeddings / original)              */
    double low_freq_factor, high_freq_factor; /* llama3                                              */
    int    original_max_position_embeddings;  /* llama3, longrope, yarn                              */
    int    max_position_embeddings;           /* longrope and yarn: derives the attention factor     */
    const double* short_factor;               /* longrope: host, r/2 values (per-pair divisors)      */
    const double* long_factor;                /* longrope: host, r/2 values                          */
    double attention_factor;                  /* <= 0: derive (1; longrope sqrt(1 + ln s / ln orig)  */
                                              /*   with s = max / orig; yarn 0.1 ln s + 1)           */
    double beta_fast, beta_slow;              /* yarn: <= 0 means 32 and 1                           */
    double mscale, mscale_all_dim;            /* yarn: both > 0 selects the ratio form               */
    int    truncate;                          /* yarn: nonzero rounds the ramp ends outwards         */
} da_rope_scaling;

/* The per-layer switches of the attention step (page 1, DecoderConfig / DecoderAttention.__init__). */
typedef struct {
    int         dtype;                        /* da_dtype of q, k, v, q_rot, caches and out          */
    int         head_dim;                     /* d: 64 or 128                                        */
    int         num_attention_heads;          /* Hq                                                   */
    int         num_key_value_heads;          /* Hkv, divides Hq                                      */
    int         rotary_dim;                   /* r: even, 2 <= r <= d                                 */
    const float* q_norm_w;                    /* device [d] fp32, or NULL for no q/k norm (the pages: */
    const float* k_norm_w;                    /*   "absent, not identity"); both or neither          */
    double      eps;                          /* RMSNorm epsilon                                      */
    int         window;                       /* sliding window w >= 0 (0 = full attention)           */
    float       softcap;                      /* logit soft-cap c >= 0: z -> c tanh(z / c); 0 = off    */
    float       scale;                        /* softmax scale; 0 means 1/sqrt(d)                     */
    const float* sinks;                       /* device [Hq] fp32 learned sink logits, or NULL (page  */
                                              /*   "Model resolution", gpt_oss: one extra logit per   */
                                              /*   head in every query's softmax, its share dropped;  */
                                              /*   in the units of the scaled, capped scores, not     */
                                              /*   capped itself, seen whatever the window)           */
} da_layer;

/*
 * da_rope_tables_build -- cos/sin of each token's rotation angles (page 1, "Scaled RoPE": rope_inv_freq
 * and rope_tables).
 *
 * Frequencies inv_i (i < r/2) follow rs->kind; for token t at position p = positions[t]:
 *     cos[t, i] = cos(p * inv_i) * af,   sin[t, i] = sin(p * inv_i) * af
 * The angle p * inv_i is formed in fp64 and reduced modulo 2 pi before the fp32 sine/cosine.
 * LongRoPE picks its long table for a token whose sequence length seq_len[t] (the total length of its
 * sequence after this step) exceeds original_max_position_embeddings, its short table otherwise.
 *
 *   positions  device int32 [n], each >= 0
 *   seq_len    device int32 [n]; required for DA_ROPE_LONGROPE, ignored (may be NULL) otherwise
 *   cos, sin   device fp32 [n, r/2], written
 * Errors: DA_ERR_INVALID_ARG (NULL pointers, n < 0, bad theta/factors/rotary_dim, missing longrope tables),
 *         DA_ERR_UNSUPPORTED (unknown kind). n == 0 enqueues nothing.
 */
int da_rope_tables_build(const da_rope_scaling* rs, const int32_t* positions, const int32_t* seq_len,
                         int n, float* cos, float* sin, cudaStream_t stream);

/*
 * da_kv_cache_update -- per-head q/k RMSNorm (when the layer has norm weights), RoPE on q and k, and the
 * cache write (page 1, DecoderAttention.forward: q_norm/k_norm, apply_rope, cache.update(layer, k, v,
 * positions, rows); page "MoE, optimisers, decoding", §3.3 KVCache.update and §4 Rotary).
 *
 * For each token t and head:  x <- x / sqrt(mean(x^2) + eps) * w      (optional)
 *                             x'_i       = x_i c_i - x_{i+r/2} s_i     (i < r/2)
 *                             x'_{i+r/2} = x_{i+r/2} c_i + x_i s_i;    dims >= r pass through
 * then  q_rot[t] = q', k_cache[rows[t], g, positions[t], :] = k'_g, v_cache[rows[t], g, positions[t], :] = v_g
 * (v copied bit for bit). Arithmetic in fp32; bf16 outputs are rounded to nearest even.
 *
 *   q, k, v       device [N, Hq, d], [N, Hkv, d], [N, Hkv, d]
 *   rows          device int32 [n], each in [0, num_rows)
 *   positions     device int32 [n], each in [0, max_len)
 *   cos, sin      device fp32 [n, r/2] from da_rope_tables_build
 *   q_rot         device [N, Hq, d], written; may be the same buffer as q
 *   k_cache, v_cache  device [num_rows, Hkv, max_len, d], written at the (row, position) slots only
 * Every pointer, cos/sin and the norm weights included, must be 16-byte aligned (16-byte vector accesses).
 * Two tokens of one call must not name the same (row, position). A token whose row or position is out of
 * range is skipped and sets DA_ERR_DEVICE_INDEX on the device.
 */
int da_kv_cache_update(const da_layer* layer, const void* q, const void* k, const void* v, int n,
                       const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                       void* q_rot, void* k_cache, void* v_cache, int num_rows, int max_len,
                       cudaStream_t stream);

/*
 * da_kv_cache_update_rope -- da_kv_cache_update with the rotation's cos/sin formed inside the kernel from
 * each token's position (and seq_len, for LongRoPE's table switch) by the same arithmetic as
 * da_rope_tables_build, so the outputs are the same bits as da_rope_tables_build followed by
 * da_kv_cache_update, without the tables' round trip through memory or their launch.
 *
 *   rs         the layer's rotary scaling; rs->rotary_dim must equal layer->rotary_dim
 *   seq_len    device int32 [n]; required for DA_ROPE_LONGROPE, ignored (may be NULL) otherwise
 *   the rest   as for da_kv_cache_update (a position < 0 rotates by zero and sets DA_ERR_DEVICE_INDEX)
 * Errors: as da_rope_tables_build and da_kv_cache_update; DA_ERR_UNSUPPORTED unless the layer is bf16 with
 *         head_dim 128 and rotary_dim a multiple of 16 (use the two calls otherwise).
 */
int da_kv_cache_update_rope(const da_layer* layer, const da_rope_scaling* rs, const void* q, const void* k,
                            const void* v, int n, const int32_t* rows, const int32_t* positions,
                            const int32_t* seq_len, void* q_rot, void* k_cache, void* v_cache, int num_rows,
                            int max_len, cudaStream_t stream);

/*
 * da_attn_prefill -- causal GQA attention of prefill chunks over their cache rows (page 1,
 * DecoderAttention.forward: window_mask then causal_attention; "Model resolution" for soft-capping).
 *
 * Sequence b owns tokens q_start[b] .. q_start[b+1]-1 of q_rot/out, at positions first_pos[b] + i, and
 * reads cache row rows[b]. Its keys are slots 0 .. first_pos[b] + n_b - 1 of that row (the chunk's own keys
 * must already be written, e.g. by da_kv_cache_update). For query head h with KV head g:
 *     z_j = scale * q_rot[t, h] . k_cache[row, g, j];   z_j = c tanh(z_j / c) when softcap c > 0
 *     out[t, h] = sum_j softmax(z)_j v_cache[row, g, j]   over the visible j; 0 if none is visible
 * With layer->sinks, head h's softmax also takes the logit sinks[h] (page "Model resolution", gpt_oss):
 *     out[t, h] = sum_j e^(z_j - m) v_j / (sum_j e^(z_j - m) + e^(sinks[h] - m)),  m = max(max_j z_j, sinks[h])
 * bf16 layers run on the tcgen05 tensor cores (bf16 operands, fp32 accumulation and softmax); fp32 layers
 * and calls with key_positions run a CUDA-core kernel in fp32.
 *
 *   q_rot          device [N, Hq, d];  n_tokens = N (= q_start[S]); rows past N are never read
 *   n_seqs         number of chunks S >= 0
 *   q_start        device int32 [S+1], nondecreasing, q_start[0] = 0
 *   rows           device int32 [S];  first_pos  device int32 [S]
 *   max_q_len      host int >= every chunk length (sizes the grid; chunks past it are not computed)
 *   key_positions  device int32 [num_rows, max_len] or NULL. NULL: slot j holds position j. Otherwise slot j
 *                  of a row holds the key at position key_positions[row, j] (negative = empty slot) and every
 *                  slot of the row is scanned.
 *   out            device [N, Hq, d], written for the chunks' tokens
 *   workspace, ws_bytes  unused by prefill (pass NULL, 0)
 * Caches must hold finite values in slots that a chunk reads; unwritten slots past a row's length are never
 * allowed to affect the result.
 */
int da_attn_prefill(const da_layer* layer, const void* q_rot, int n_tokens, const void* k_cache, const void* v_cache,
                    int num_rows, int max_len, int n_seqs, const int32_t* q_start, const int32_t* rows,
                    const int32_t* first_pos, int max_q_len, const int32_t* key_positions, void* out,
                    void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * da_attn_decode -- one new token per sequence attends over its cache row (the decode case of
 * DecoderAttention.forward, page 1; a window bounds the keys read to w, page 1 "Sliding windows").
 *
 * Sequence s has one query q_rot[s] at position positions[s] in row rows[s]; it sees slots
 * 0 .. positions[s] (its own key must already be written). Same arithmetic as da_attn_prefill. The bf16
 * path splits the keys of each (sequence, KV head) into chunks processed in parallel, each chunk's partial
 * softmax (max, sum, weighted values) going to `workspace`, then merges them in a fixed order (results
 * are deterministic run to run).
 *
 *   q_rot      device [S, Hq, d];  rows, positions  device int32 [S]
 *   key_positions  as in da_attn_prefill, or NULL
 *   out        device [S, Hq, d]
 *   workspace  device scratch of at least da_decode_workspace_bytes(layer, n_seqs, max_len) bytes,
 *              16-byte aligned; its contents need no initialisation and are clobbered
 */
int da_attn_decode(const da_layer* layer, const void* q_rot, const void* k_cache, const void* v_cache,
                   int num_rows, int max_len, int n_seqs, const int32_t* rows, const int32_t* positions,
                   const int32_t* key_positions, void* out, void* workspace, size_t ws_bytes,
                   cudaStream_t stream);

/* Scratch bytes da_attn_decode needs for n_seqs sequences over a cache of max_len positions per row
 * (0 when the layer is invalid or decode needs none). Pure host arithmetic. */
size_t da_decode_workspace_bytes(const da_layer* layer, int n_seqs, int max_len);

/*
 * da_attn_mixed -- da_attn_prefill and da_attn_decode of one layer's mixed batch (prefill chunks and decode
 * tokens in the same step, as DecoderAttention.forward on page 1 takes a batch of both) in one call, the two
 * running side by side on the GPU.
 *
 * Token layout of q_rot and out: the chunks' tokens first (rows 0 .. n_tokens-1, as da_attn_prefill takes
 * them), then one token per decoding sequence (rows n_tokens .. n_tokens + n_decode - 1, as da_attn_decode).
 * The results are bit for bit those of da_attn_prefill followed by da_attn_decode with the same arguments:
 * the same kernels compute every output, and no output depends on how the GPU is shared.
 *
 * When both parts run on the tensor-core paths (bf16, d = 128, no key_positions) and both work hints are
 * positive, the prefill's persistent grid is given part of the SMs and the decode's blocks the rest, so that
 * the compute-bound prefill and the memory-bound decode overlap. The split minimises the modelled time of the
 * two on this GPU (prefill ~7.2 TFLOP/s per SM, 0.8 of that over a paged pool; decode ~100 GB/s per SM up to
 * ~7.2 TB/s in all), and the call runs the two one after the other on `stream` when that model says overlap
 * does not pay (by 3% or more). To overlap, the call forks onto a stream the library owns (created, with two
 * events, on the first such call on each device and kept until the process exits) and joins back to `stream`
 * before returning: work enqueued on `stream` afterwards sees both results. Calls from several host threads
 * are serialised while they enqueue. The fork and join are capturable into a CUDA graph; make the first
 * overlapping call on each device (the one that creates the stream and events) outside any capture.
 *
 *   n_tokens, n_seqs, q_start, chunk_rows, first_pos, max_q_len   the prefill part, as da_attn_prefill
 *   n_decode, dec_rows, dec_positions                             the decode part, as da_attn_decode
 *   prefill_pairs  host hint: visible (query, key) pairs summed over the chunks' tokens (one query head);
 *                  0 when unknown (then the parts run one after the other)
 *   decode_keys    host hint: visible keys summed over the decode tokens; 0 when unknown
 *   workspace, ws_bytes  decode scratch of at least da_decode_workspace_bytes(layer, n_decode, max_len)
 * Errors: every check of both calls, made before anything is enqueued.
 */
int da_attn_mixed(const da_layer* layer, const void* q_rot, const void* k_cache, const void* v_cache, int num_rows,
                  int max_len, int n_tokens, int n_seqs, const int32_t* q_start, const int32_t* chunk_rows,
                  const int32_t* first_pos, int max_q_len, int n_decode, const int32_t* dec_rows,
                  const int32_t* dec_positions, double prefill_pairs, double decode_keys, void* out, void* workspace,
                  size_t ws_bytes, cudaStream_t stream);

/*
 * da_attn_decode_noalloc -- da_attn_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this entry point exists for callers of this library that may not call
 * cudaMalloc or any allocating routine -- for example a host process whose device memory is owned by
 * another component's pool, or a path where an allocation's implicit synchronisation is not acceptable.
 * It computes exactly what da_attn_decode computes (same arguments, minus the workspace) and allocates
 * nothing: the split-K partials go to a fixed scratch array of da_decode_noalloc_max_scratch_bytes()
 * bytes (32 MiB) in the library's own device memory, which every GPU that loads the library holds until
 * the process exits.
 *  - A call whose split plan needs more scratch than that (da_decode_workspace_bytes(layer, n_seqs,
 *    max_len) > 32 MiB) returns DA_ERR_INVALID_ARG and enqueues nothing; split the batch or use
 *    da_attn_decode.
 *  - Every call shares the one array: calls whose kernels overlap on the GPU (different streams, or
 *    different threads without ordering) race on it and may return wrong results. Calls on one stream are
 *    ordered and safe. The scratch needs no clearing between calls: each call writes every partial before
 *    reading it.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress) with that
 *    device current; make that first call before any stream capture.
 */
int da_attn_decode_noalloc(const da_layer* layer, const void* q_rot, const void* k_cache, const void* v_cache,
                           int num_rows, int max_len, int n_seqs, const int32_t* rows, const int32_t* positions,
                           const int32_t* key_positions, void* out, cudaStream_t stream);

/* Size in bytes of the fixed scratch behind da_attn_decode_noalloc. */
size_t da_decode_noalloc_max_scratch_bytes(void);

/*
 * Paged KV pool (page 1, "Sliding windows": the engine keeps keys and values in fixed-size blocks that each
 * request maps through its own block table, so that blocks every query has moved past can be recycled).
 * Position p of cache row r lives in block block_table[r * max_blocks + p / block_size], at offset
 * p % block_size:  k_pool[block, g, p % block_size, :] is key head g of that position.
 */
typedef struct {
    void*          k_pool;        /* device [n_blocks, Hkv, block_size, d], 16-byte aligned                 */
    void*          v_pool;        /* device [n_blocks, Hkv, block_size, d], 16-byte aligned                 */
    int            n_blocks;      /* blocks in each pool, >= 1 (n_blocks * Hkv * block_size < 2^31)         */
    int            block_size;    /* positions per block, >= 1; the bf16 tensor-core paths need a multiple  */
                                  /*   of 64 (other sizes run the CUDA-core kernel)                         */
    const int32_t* block_table;   /* device int32 [num_rows, max_blocks]; an entry outside [0, n_blocks)    */
                                  /*   (e.g. -1 for a recycled block) maps nothing                          */
    int            num_rows;      /* cache rows (requests), >= 1                                            */
    int            max_blocks;    /* entries per row: a row holds positions < max_blocks * block_size       */
} da_paged_kv;

/*
 * da_kv_cache_update_paged -- da_kv_cache_update into a paged pool: token t's k_rot and v go to the slot of
 * (rows[t], positions[t]) that kv->block_table names. A token whose row or position is out of range, or
 * whose block is unmapped, writes nothing and sets the device error word (DA_ERR_DEVICE_INDEX).
 */
int da_kv_cache_update_paged(const da_layer* layer, const void* q, const void* k, const void* v, int n,
                             const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                             void* q_rot, const da_paged_kv* kv, cudaStream_t stream);

/* da_kv_cache_update_rope_paged -- da_kv_cache_update_rope into a paged pool (as da_kv_cache_update_paged). */
int da_kv_cache_update_rope_paged(const da_layer* layer, const da_rope_scaling* rs, const void* q, const void* k,
                                  const void* v, int n, const int32_t* rows, const int32_t* positions,
                                  const int32_t* seq_len, void* q_rot, const da_paged_kv* kv, cudaStream_t stream);

/*
 * da_attn_prefill_paged -- da_attn_prefill over a paged pool (same arithmetic, sinks included). A chunk reads
 * positions from its oldest query's first visible key (first_pos - w + 1 with a window w, else 0) to its
 * last token; blocks wholly before that may be unmapped. A visible position without a block sets the device
 * error word (its keys are then not the caller's).
 */
int da_attn_prefill_paged(const da_layer* layer, const void* q_rot, int n_tokens, const da_paged_kv* kv, int n_seqs,
                          const int32_t* q_start, const int32_t* rows, const int32_t* first_pos, int max_q_len,
                          void* out, cudaStream_t stream);

/*
 * da_attn_decode_paged -- da_attn_decode over a paged pool. On the split-K path the chunks of a sequence
 * start at its first visible key rounded down to a 64-key tile (a tile never straddles two blocks), so the
 * workspace is sized by da_decode_workspace_bytes_paged.
 */
int da_attn_decode_paged(const da_layer* layer, const void* q_rot, const da_paged_kv* kv, int n_seqs,
                         const int32_t* rows, const int32_t* positions, void* out, void* workspace, size_t ws_bytes,
                         cudaStream_t stream);

/* How many SMs da_attn_mixed (contiguous caches) gives the prefill's persistent grid, for these hints, on a GPU
 * of n_sm SMs: n_sm
 * when the two parts would run one after the other. Pure host arithmetic (the model described at
 * da_attn_mixed), for callers that plan batches and for tests. DA_ERR_INVALID_ARG (negative) for an invalid
 * layer, n_sm < 1, or hints that are negative or not finite. */
int da_attn_mixed_prefill_sms(const da_layer* layer, int n_sm, double prefill_pairs, double decode_keys);

/* da_attn_mixed over a paged pool (the prefill and decode parts as da_attn_prefill_paged and
 * da_attn_decode_paged; workspace per da_decode_workspace_bytes_paged). */
int da_attn_mixed_paged(const da_layer* layer, const void* q_rot, const da_paged_kv* kv, int n_tokens, int n_seqs,
                        const int32_t* q_start, const int32_t* chunk_rows, const int32_t* first_pos, int max_q_len,
                        int n_decode, const int32_t* dec_rows, const int32_t* dec_positions, double prefill_pairs,
                        double decode_keys, void* out, void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes da_attn_decode_paged needs for n_seqs sequences of a pool whose rows hold max_positions
 * (= max_blocks * block_size) positions (0 when the layer is invalid or decode needs none). Host arithmetic. */
size_t da_decode_workspace_bytes_paged(const da_layer* layer, int n_seqs, int max_positions);

/*
 * Multi-head latent attention, absorbed form (page 1, "Multi-head latent attention" and "Serving it:
 * absorbing the up-projections"). Each token caches one row [c, k_rope] of kv_lora_rank + qk_rope_dim bf16
 * numbers; each query head arrives mapped into latent space, q = [W_uk^T q_nope, q_rope], and decode is
 * multi-query attention of all heads over the rows, whose first kv_lora_rank features are the values. The
 * output is each head's latent (kv_lora_rank wide); W_uv and o_proj are applied by the caller.
 * Supported: bf16, kv_lora_rank 512, qk_rope_dim 64 (DeepSeek-V2/V3, Kimi K2), num_heads a multiple of 8.
 */
typedef struct {
    int   num_heads;       /* query heads sharing each latent row                                       */
    int   kv_lora_rank;    /* latent (= value) width: 512                                              */
    int   qk_rope_dim;     /* rotary width: 64                                                         */
    float scale;           /* softmax scale: (qk_nope_head_dim + qk_rope_dim)^-0.5, times YaRN's squared */
                           /*   temperature (0.1 mscale_all_dim ln s + 1)^2 when rope_scaling sets it  */
    int   window;          /* 0 = full attention                                                       */
} da_mla_layer;

/*
 * da_mla_cache_update -- writes token t's row [latent[t], rope(k_rope[t])] at (rows[t], positions[t]) and,
 * when q is not NULL, rotates the last qk_rope_dim features of every head of q[t] in place. The rotary
 * inputs are in DeepSeek's adjacent-pair order (x[2i], x[2i+1]); they are deinterleaved (evens, then odds)
 * and rotated by the split-half rotation with cos/sin [n, qk_rope_dim / 2] from da_rope_tables_build:
 * y'[i] = x[2i] c_i - x[2i+1] s_i, y'[i + r/2] = x[2i+1] c_i + x[2i] s_i.
 *   latent [n, 512], k_rope [n, 64], q [n, H, 576] or NULL, cache [num_rows, max_len, 576] (device, bf16,
 *   16-byte aligned). A token whose slot is out of range writes nothing and sets DA_ERR_DEVICE_INDEX.
 */
int da_mla_cache_update(const da_mla_layer* layer, const void* latent, const void* k_rope, int n, const int32_t* rows,
                        const int32_t* positions, const float* cos, const float* sin, void* q, void* cache, int num_rows,
                        int max_len, cudaStream_t stream);

/*
 * da_mla_decode -- one query token per sequence: out[s, h] = sum_j softmax_j(scale q[s,h] . row_j) row_j[:512]
 * over rows 0 .. positions[s] of cache row rows[s] (the last w with a window). Split-K with a fixed-order
 * merge (deterministic); the workspace is sized by da_mla_workspace_bytes.
 *   q [S, H, 576], cache [num_rows, max_len, 576], out [S, H, 512] (device, bf16, 16-byte aligned).
 */
int da_mla_decode(const da_mla_layer* layer, const void* q, const void* cache, int num_rows, int max_len, int n_seqs,
                  const int32_t* rows, const int32_t* positions, void* out, void* workspace, size_t ws_bytes,
                  cudaStream_t stream);
size_t da_mla_workspace_bytes(const da_mla_layer* layer, int n_seqs, int max_len);

/* The same over a paged pool of latent rows: kv->k_pool [n_blocks, 1, block_size, 576] (v_pool unused; the
 * page's pool passes one tensor as both); block_size a multiple of 64 for da_mla_decode_paged. The
 * workspace is sized by da_mla_workspace_bytes_paged(layer, n_seqs, max_blocks * block_size). */
int da_mla_cache_update_paged(const da_mla_layer* layer, const void* latent, const void* k_rope, int n,
                              const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                              void* q, const da_paged_kv* kv, cudaStream_t stream);
int da_mla_decode_paged(const da_mla_layer* layer, const void* q, const da_paged_kv* kv, int n_seqs,
                        const int32_t* rows, const int32_t* positions, void* out, void* workspace, size_t ws_bytes,
                        cudaStream_t stream);
size_t da_mla_workspace_bytes_paged(const da_mla_layer* layer, int n_seqs, int max_positions);

/* MLAAttention's softmax scale (page 1, MLAAttention.__init__): (qk_nope_head_dim + qk_rope_head_dim)^-0.5,
 * times (0.1 mscale_all_dim ln factor + 1)^2 when mscale_all_dim > 0 and factor > 1 (YaRN's temperature);
 * pass 0 for either to leave it out. Host arithmetic; NaN for non-positive head dims. */
double da_mla_softmax_scale(int qk_nope_head_dim, int qk_rope_head_dim, double factor, double mscale_all_dim);

/*
 * da_qkv_project_update -- the projection before the step fused with the step's first half (page 1,
 * DecoderAttention.forward: q_proj/k_proj/v_proj, q_norm/k_norm, apply_rope, cache.update): for token t,
 *     y = x[t] W_qkv^T (+ bias),  W_qkv = [q_proj; k_proj; v_proj] stacked by rows ([(Hq + 2 Hkv) d, hidden])
 * then for each q and k head the layer's RMSNorm (when it has norm weights) and RoPE with cos/sin[t] (from
 * da_rope_tables_build), written to q_rot[t] and to the token's cache slot, and each v head to its slot; the
 * q/k/v intermediate never reaches memory. One tcgen05 GEMM whose epilogue does the rest (fp32 until the
 * bf16 stores). Supported: bf16, head_dim 128, rotary_dim 128, Hq + 2 Hkv even, hidden a multiple of 64.
 *   x [n, hidden], w_qkv as above (device bf16, 16-byte aligned), bias [(Hq + 2 Hkv) d] fp32 or NULL; the other
 *   arguments as for da_kv_cache_update (same slot rules and device error reporting).
 */
int da_qkv_project_update(const da_layer* layer, const void* x, const void* w_qkv, const float* bias, int n, int hidden,
                          const int32_t* rows, const int32_t* positions, const float* cos, const float* sin,
                          void* q_rot, void* k_cache, void* v_cache, int num_rows, int max_len, cudaStream_t stream);
int da_qkv_project_update_paged(const da_layer* layer, const void* x, const void* w_qkv, const float* bias, int n,
                                int hidden, const int32_t* rows, const int32_t* positions, const float* cos,
                                const float* sin, void* q_rot, const da_paged_kv* kv, cudaStream_t stream);

/*
 * da_linear -- y = x w^T (+ bias) with x [m, k], w [n, k], y [m, n] bf16 (fp32 accumulation, bias fp32 [n] or
 * NULL): the o_proj after the step (page 1, DecoderAttention.forward), on the same tcgen05 GEMM. n a multiple
 * of 256, k a multiple of 64; pointers 16-byte aligned.
 */
int da_linear(const void* x, const void* w, const float* bias, int m, int n, int k, void* y, cudaStream_t stream);

/*
 * Block manager of a paged pool (host bookkeeping only; page 1, "Sliding windows": each request maps pool
 * blocks through its own block table, and a group of windowed layers keeps its own table so that the blocks
 * every query has moved past are recycled: a windowed-only request holds at most ceil(w / block_size) + 1
 * blocks however long its context). One pool serves one layer group (one window w, 0 = full attention) and
 * owns the host copy of that group's table [num_rows, max_blocks] (-1 = no block); the device pools and the
 * device copy of the table belong to the caller, who copies the table after the calls that change it. Free
 * blocks are handed out last-freed first. A pool is not thread-safe.
 */
typedef struct da_block_pool da_block_pool;

/* A pool of n_blocks blocks of block_size positions for num_rows rows of max_blocks table entries each,
 * for layers with window `window` (0 = full). NULL on invalid arguments or allocation failure. */
da_block_pool* da_block_pool_create(int n_blocks, int block_size, int num_rows, int max_blocks, int window);
void da_block_pool_destroy(da_block_pool* pool);

/*
 * Before a step that attends from position first_pos (the row's oldest query in the step) up to position
 * length - 1 (its newest token): maps every block of positions [lo, length) that is not yet mapped, with
 * lo = max(0, first_pos - w + 1) for a windowed pool and 0 otherwise, and (windowed pools) releases the
 * row's blocks that lie wholly before lo. All or nothing: DA_ERR_OUT_OF_BLOCKS leaves the pool unchanged.
 * first_pos must not decrease for a row until the row is released. DA_ERR_INVALID_ARG for a bad row,
 * first_pos < 0, length < first_pos, or length beyond max_blocks * block_size.
 */
int da_block_pool_reserve(da_block_pool* pool, int row, int first_pos, int length);

/* Releases every block of a row (its request has finished); the row can then serve a new request. */
int da_block_pool_release(da_block_pool* pool, int row);

/* Free blocks (-1 for a NULL pool). */
int da_block_pool_free_blocks(const da_block_pool* pool);

/* Blocks a row holds after da_block_pool_reserve(pool, row, first_pos, length) (-1 on bad arguments). */
int da_block_pool_blocks_needed(const da_block_pool* pool, int first_pos, int length);

/* The host block table [num_rows, max_blocks], owned by the pool; valid until the pool is destroyed. */
const int32_t* da_block_pool_table(const da_block_pool* pool);

/* Waits for `stream`, then reads and clears the device error word that kernels set on an out-of-range
 * index (DA_ERR_DEVICE_INDEX) or a bounded wait that gave up (DA_ERR_TIMEOUT). Returns DA_OK when clear,
 * DA_ERR_CUDA if the wait itself failed. */
int da_check_device_error(cudaStream_t stream);

/* Message for the last nonzero return on the calling thread ("" if none). Owned by the library. */
const char* da_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int da_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DECATTN_H */
