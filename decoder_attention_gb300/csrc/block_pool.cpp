// Host-side block manager of a paged KV pool (page 1, "Sliding windows": each request maps the blocks of a
// shared pool through its own block table; a group of windowed layers gets its own table so that the blocks
// every query has moved past can be recycled; a windowed-only request then holds ceil(w / block) + 1 blocks
// however long its context).
//
// One da_block_pool serves one layer group (one window). It owns the host copy of the group's block table
// [num_rows, max_blocks]; the device pools and the device copy of the table are the caller's (copy the
// table after the calls that change it). Free blocks form a stack, so a recycled block is the next one
// handed out. Not thread-safe: one pool, one caller thread.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "decattn.h"

struct da_block_pool {
  int n_blocks, block_size, num_rows, max_blocks, window;
  std::vector<int32_t> table;   // [num_rows * max_blocks], -1 = no block
  std::vector<int32_t> free_;   // stack of free block ids
  std::vector<int32_t> lo;      // per row: first block index still mapped (blocks before it were released)
  std::vector<int32_t> hi;      // per row: one past the last block index mapped
};

namespace {

// Block indices [b0, b1) that a row must map for queries from position first_pos on, and up to length.
void needed_range(const da_block_pool* p, int first_pos, int length, int& b0, int& b1) {
  const int lo_pos = p->window > 0 ? (first_pos - p->window + 1 > 0 ? first_pos - p->window + 1 : 0) : 0;
  b0 = lo_pos / p->block_size;
  b1 = (length + p->block_size - 1) / p->block_size;
}

}  // namespace

extern "C" {

da_block_pool* da_block_pool_create(int n_blocks, int block_size, int num_rows, int max_blocks, int window) {
  if (n_blocks < 1 || block_size < 1 || num_rows < 1 || max_blocks < 1 || window < 0) return nullptr;
  if (static_cast<long long>(num_rows) * max_blocks > (1LL << 31) - 1) return nullptr;
  da_block_pool* p = new (std::nothrow) da_block_pool;
  if (!p) return nullptr;
  p->n_blocks = n_blocks;
  p->block_size = block_size;
  p->num_rows = num_rows;
  p->max_blocks = max_blocks;
  p->window = window;
  try {
    p->table.assign(static_cast<size_t>(num_rows) * max_blocks, -1);
    p->free_.resize(n_blocks);
    for (int i = 0; i < n_blocks; ++i) p->free_[i] = n_blocks - 1 - i;   // block 0 on top
    p->lo.assign(num_rows, 0);
    p->hi.assign(num_rows, 0);
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void da_block_pool_destroy(da_block_pool* p) { delete p; }

int da_block_pool_reserve(da_block_pool* p, int row, int first_pos, int length) {
  if (!p || row < 0 || row >= p->num_rows || first_pos < 0 || length < first_pos) return DA_ERR_INVALID_ARG;
  int b0, b1;
  needed_range(p, first_pos, length, b0, b1);
  if (b1 > p->max_blocks) return DA_ERR_INVALID_ARG;
  int32_t* t = p->table.data() + static_cast<size_t>(row) * p->max_blocks;
  // a window only moves forward: blocks of this row before b0 are released first, then the missing ones in
  // [b0, b1) are mapped (all or none)
  int missing = 0;
  for (int b = b0 > p->lo[row] ? b0 : p->lo[row]; b < b1; ++b) missing += t[b] < 0;
  int releasable = 0;
  if (p->window > 0)
    for (int b = p->lo[row]; b < b0 && b < p->hi[row]; ++b) releasable += t[b] >= 0;
  if (missing > static_cast<int>(p->free_.size()) + releasable) return DA_ERR_OUT_OF_BLOCKS;
  if (p->window > 0) {
    for (int b = p->lo[row]; b < b0 && b < p->hi[row]; ++b)
      if (t[b] >= 0) {
        p->free_.push_back(t[b]);
        t[b] = -1;
      }
    if (b0 > p->lo[row]) p->lo[row] = b0;
  }
  for (int b = p->lo[row]; b < b1; ++b)
    if (t[b] < 0) {
      t[b] = p->free_.back();
      p->free_.pop_back();
    }
  if (b1 > p->hi[row]) p->hi[row] = b1;
  return DA_OK;
}

int da_block_pool_release(da_block_pool* p, int row) {
  if (!p || row < 0 || row >= p->num_rows) return DA_ERR_INVALID_ARG;
  int32_t* t = p->table.data() + static_cast<size_t>(row) * p->max_blocks;
  for (int b = 0; b < p->hi[row]; ++b)
    if (t[b] >= 0) {
      p->free_.push_back(t[b]);
      t[b] = -1;
    }
  p->lo[row] = p->hi[row] = 0;
  return DA_OK;
}

int da_block_pool_free_blocks(const da_block_pool* p) { return p ? static_cast<int>(p->free_.size()) : -1; }

int da_block_pool_blocks_needed(const da_block_pool* p, int first_pos, int length) {
  if (!p || first_pos < 0 || length < first_pos) return -1;
  int b0, b1;
  needed_range(p, first_pos, length, b0, b1);
  return b1 - b0;
}

const int32_t* da_block_pool_table(const da_block_pool* p) { return p ? p->table.data() : nullptr; }

}  // extern "C"
