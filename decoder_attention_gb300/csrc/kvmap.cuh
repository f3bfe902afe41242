// Device-side addressing of cache slots, contiguous or paged (one block table per cache row).
#pragma once

#include "internal.h"

namespace da {

template <typename Args>
__device__ __forceinline__ KvLayout kv_layout(const Args& a) {
  KvLayout L;
  L.block_table = a.block_table;
  L.num_rows = a.num_rows;
  L.max_len = a.max_len;
  L.hkv = a.hkv;
  L.block_size = a.block_size;
  L.max_blocks = a.max_blocks;
  L.n_blocks = a.n_blocks;
  return L;
}

// Cache row (in units of d elements) of (row, KV head 0, position pos), or -1 when the slot is outside the
// cache (row or position out of range, or a paged row whose block for pos is missing). KV head g adds
// g * kv_head_stride(L).
__device__ __forceinline__ long long kv_slot(const KvLayout& L, int row, int pos) {
  if (row < 0 || row >= L.num_rows || pos < 0 || pos >= L.max_len) return -1;
  if (L.block_table == nullptr) return static_cast<long long>(row) * L.hkv * L.max_len + pos;
  const int b = L.block_table[static_cast<long long>(row) * L.max_blocks + pos / L.block_size];
  if (b < 0 || b >= L.n_blocks) return -1;
  return static_cast<long long>(b) * L.hkv * L.block_size + pos % L.block_size;
}

__device__ __forceinline__ long long kv_head_stride(const KvLayout& L) {
  return L.block_table ? L.block_size : L.max_len;
}

}  // namespace da
