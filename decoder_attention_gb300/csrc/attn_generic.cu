// CUDA-core attention in fp32 for any layer the tensor-core kernels do not take: fp32 caches (the
// fp32 path), explicit key positions, head widths or GQA groups outside the fast kernels' range.
//
// Computes, per query token and head, what causal_attention computes in DecoderAttention.forward
// (page "42. More models: ...", sections "What differs between model families" and "Sliding windows"):
// softmax over the visible keys of scale * q.k (soft-capped when a cap is set), weighted sum of values.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "kvmap.cuh"

namespace da {

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }
template <typename T>
__device__ __forceinline__ void st_elem(T* p, float v);
template <>
__device__ __forceinline__ void st_elem<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_elem<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Block = 4 warps for one (query token, query head). Warps take keys round-robin; within a warp each lane
// owns D/32 components. Online softmax per warp, merged through shared memory at the end.
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_generic_kernel(const AttnArgs a) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int i = blockIdx.x;
  __shared__ float sm_m[4], sm_l[4];
  __shared__ float sm_o[4][D];
  pdl_wait();   // inputs written by the stream's previous kernel are visible

  int t, p, kv_len;
  if (a.q_start) {
    const int t0 = a.q_start[s], t1 = a.q_start[s + 1];
    if (i >= t1 - t0) return;
    t = t0 + i;
    p = a.first_pos[s] + i;
    kv_len = a.first_pos[s] + (t1 - t0);
  } else {
    t = s;
    p = a.positions[s];
    kv_len = p + 1;
  }
  const int row = a.rows[s];
  const int group = a.hq / a.hkv;
  const int g = h / group;
  T* out = static_cast<T*>(a.out) + (static_cast<long long>(t) * a.hq + h) * D;
  if (row < 0 || row >= a.num_rows || p < 0 || (a.key_positions == nullptr && kv_len > a.max_len)) {
    if (threadIdx.x == 0) set_error(a.err, kErrIndex);
    for (int e = threadIdx.x; e < D; e += blockDim.x) st_elem<T>(out + e, 0.f);
    return;
  }

  const T* qv = static_cast<const T*>(a.q_rot) + (static_cast<long long>(t) * a.hq + h) * D;
  float q[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) q[j] = ld_elem<T>(qv + lane + 32 * j);

  const KvLayout kvl = kv_layout(a);
  const long long plane = (static_cast<long long>(row) * a.hkv + g) * a.max_len;   // contiguous caches
  const long long head_off = g * kv_head_stride(kvl);                                   // paged pools
  const T* kb = static_cast<const T*>(a.k_cache);
  const T* vb = static_cast<const T*>(a.v_cache);
  const float scale = a.scale;

  int j_lo = 0, j_hi;
  if (a.key_positions == nullptr) {
    j_hi = min(p + 1, kv_len);
    if (a.window > 0) j_lo = max(0, p - a.window + 1);
  } else {
    j_hi = a.max_len;
  }
  const int32_t* kp = a.key_positions ? a.key_positions + static_cast<long long>(row) * a.max_len : nullptr;

  float m = -CUDART_INF_F, l = 0.f;
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;

  for (int j = j_lo + warp; j < j_hi; j += 4) {
    if (kp) {
      const int kpos = kp[j];
      if (kpos < 0 || kpos > p || (a.window > 0 && p - kpos > a.window - 1)) continue;
    }
    long long kslot = plane + j;
    if (a.block_table) {
      kslot = kv_slot(kvl, row, j);
      if (kslot < 0) {   // a visible position without a block: reported, and left out
        if (lane == 0) set_error(a.err, kErrIndex);
        continue;
      }
      kslot += head_off;
    }
    const T* kr = kb + kslot * D;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) dot = fmaf(q[e], ld_elem<T>(kr + lane + 32 * e), dot);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    float z = dot * scale;
    if (a.softcap > 0.f) z = a.softcap * tanhf(z / a.softcap);
    const float m_new = fmaxf(m, z);
    const float alpha = __expf(m - m_new);   // m = -inf on the first key: alpha = 0
    const float pj = __expf(z - m_new);
    l = l * alpha + pj;
    const T* vr = vb + kslot * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = fmaf(pj, ld_elem<T>(vr + lane + 32 * e), acc[e] * alpha);
    m = m_new;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) sm_o[warp][lane + 32 * e] = acc[e];
  __syncthreads();
  float M = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_m[w]);
  const float sink = a.sinks ? a.sinks[h] : -CUDART_INF_F;   // one more logit; its share reaches no value
  M = fmaxf(M, sink);
  float L = (a.sinks && M != -CUDART_INF_F) ? __expf(sink - M) : 0.f;
  float wgt[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    wgt[w] = (sm_m[w] == -CUDART_INF_F) ? 0.f : __expf(sm_m[w] - M);
    L += wgt[w] * sm_l[w];
  }
  const float invL = L > 0.f ? 1.f / L : 0.f;
  for (int e = threadIdx.x; e < D; e += blockDim.x) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) o += wgt[w] * sm_o[w][e];
    st_elem<T>(out + e, o * invL);
  }
}

template <typename T, int D>
static cudaError_t launch_generic_t(const AttnArgs& a, cudaStream_t stream) {
  dim3 grid(a.max_q_len, a.hq, a.n_seqs);
  return launch_dependent(attn_generic_kernel<T, D>, grid, dim3(128), 0, stream, a);
}

cudaError_t launch_attn_generic(const AttnArgs& a, bool bf16, cudaStream_t stream) {
  if (a.n_seqs == 0 || a.max_q_len == 0) return cudaSuccess;
  if (bf16) return a.d == 64 ? launch_generic_t<__nv_bfloat16, 64>(a, stream) : launch_generic_t<__nv_bfloat16, 128>(a, stream);
  return a.d == 64 ? launch_generic_t<float, 64>(a, stream) : launch_generic_t<float, 128>(a, stream);
}

}  // namespace da
