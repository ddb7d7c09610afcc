// Host block allocator: free list, reference counts, copy-on-write.
//
// The block manager of the PagedAttention blog page ("SOSP 2023論文解説: vLLM",
// section "アルゴリズムの擬似コード") and of the paper summary (section 5:
// blocks are taken on demand when the last block fills and returned when the
// sequence ends; section 6: blocks are shared by reference count and a shared
// block is copied before it is written).  It never touches the GPU: it
// produces the slot of each appended token, the block tables, and the
// (src, dst) pairs that pa_copy_blocks must apply before the write.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
  };
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // taken from the back
  std::vector<int32_t> ref;
  std::unordered_map<int, Seq> seqs;

  int32_t take() {
    int32_t b = free_list.back();
    free_list.pop_back();
    ref[b] = 1;
    return b;
  }
  bool release(int32_t b) {
    if (ref[b] <= 0) return false;
    if (--ref[b] == 0) free_list.push_back(b);
    return true;
  }
};

namespace {

// Blocks that appending one token to each listed sequence would take,
// accounting for copy-on-write pairs within the batch (a copy drops a
// reference, which can let a later sequence of the same batch write in place).
int blocks_needed(const pa_alloc& a, const int* seq_ids, int n) {
  std::unordered_map<int32_t, int> ref_drop;
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const auto& sq = a.seqs.at(seq_ids[i]);
    if (sq.blocks.empty()) {
      ++need;
      continue;
    }
    const int64_t filled = sq.len - (int64_t)(sq.blocks.size() - 1) * a.block_size;
    if (filled >= a.block_size) {
      ++need;
      continue;
    }
    const int32_t last = sq.blocks.back();
    if (a.ref[last] - ref_drop[last] > 1) {
      ++need;
      ++ref_drop[last];
    }
  }
  return need;
}

}  // namespace

extern "C" {

int pa_alloc_create(int num_blocks, int block_size, pa_alloc** out) {
  if (out == nullptr || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  pa_alloc* a = new (std::nothrow) pa_alloc();
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->free_list.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) a->free_list[i] = i;
  a->ref.assign(num_blocks, 0);
  *out = a;
  return PA_OK;
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

int pa_alloc_add_seq(pa_alloc* a, int seq_id) {
  if (a == nullptr || seq_id < 0 || a->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
  a->seqs.emplace(seq_id, pa_alloc::Seq{});
  return PA_OK;
}

int pa_alloc_fork(pa_alloc* a, int parent, int child) {
  if (a == nullptr || child < 0 || !a->seqs.count(parent) || a->seqs.count(child)) return PA_ERR_INVALID_ARG;
  pa_alloc::Seq c = a->seqs.at(parent);
  for (int32_t b : c.blocks) ++a->ref[b];
  a->seqs.emplace(child, std::move(c));
  return PA_OK;
}

int pa_alloc_append_slots(pa_alloc* a, const int* seq_ids, int n, int64_t* slots_out, int32_t* copy_pairs_out,
                          int* n_pairs_out) {
  if (a == nullptr || n < 0 || (n > 0 && (seq_ids == nullptr || slots_out == nullptr))) return PA_ERR_INVALID_ARG;
  std::unordered_set<int> seen;
  for (int i = 0; i < n; ++i) {
    if (!a->seqs.count(seq_ids[i]) || !seen.insert(seq_ids[i]).second) return PA_ERR_INVALID_ARG;
  }
  if (blocks_needed(*a, seq_ids, n) > (int)a->free_list.size()) return PA_ERR_NO_FREE_BLOCKS;
  int np = 0;
  const int B = a->block_size;
  for (int i = 0; i < n; ++i) {
    auto& sq = a->seqs.at(seq_ids[i]);
    if (sq.blocks.empty()) sq.blocks.push_back(a->take());
    int64_t filled = sq.len - (int64_t)(sq.blocks.size() - 1) * B;
    if (filled >= B) {
      sq.blocks.push_back(a->take());
      filled = 0;
    } else if (a->ref[sq.blocks.back()] > 1) {
      const int32_t old_b = sq.blocks.back();
      const int32_t new_b = a->take();
      if (copy_pairs_out != nullptr) {
        copy_pairs_out[2 * np] = old_b;
        copy_pairs_out[2 * np + 1] = new_b;
      }
      ++np;
      --a->ref[old_b];
      sq.blocks.back() = new_b;
    }
    slots_out[i] = (int64_t)sq.blocks.back() * B + filled;
    ++sq.len;
  }
  if (n_pairs_out != nullptr) *n_pairs_out = np;
  return PA_OK;
}

int pa_alloc_free_seq(pa_alloc* a, int seq_id) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
  for (int32_t b : it->second.blocks) {
    if (a->ref[b] <= 0) return PA_ERR_REFCOUNT;
  }
  for (int32_t b : it->second.blocks) a->release(b);
  a->seqs.erase(it);
  return PA_OK;
}

int pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out, int cap, int* n_blocks, int* seq_len) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
  const auto& sq = it->second;
  if (n_blocks) *n_blocks = (int)sq.blocks.size();
  if (seq_len) *seq_len = (int)sq.len;
  if ((int)sq.blocks.size() > cap) return PA_ERR_INVALID_ARG;
  if (out != nullptr) std::copy(sq.blocks.begin(), sq.blocks.end(), out);
  return PA_OK;
}

int pa_alloc_block_tables(const pa_alloc* a, const int* seq_ids, int n, int max_blocks_per_seq, int32_t* tables_out,
                          int32_t* ctx_lens_out) {
  if (a == nullptr || n < 0 || max_blocks_per_seq <= 0 || (n > 0 && seq_ids == nullptr)) return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end() || (int)it->second.blocks.size() > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) {
    const auto& sq = a->seqs.at(seq_ids[i]);
    if (tables_out != nullptr) {
      int32_t* row = tables_out + (int64_t)i * max_blocks_per_seq;
      std::fill(row, row + max_blocks_per_seq, -1);
      std::copy(sq.blocks.begin(), sq.blocks.end(), row);
    }
    if (ctx_lens_out != nullptr) ctx_lens_out[i] = (int32_t)sq.len;
  }
  return PA_OK;
}

int pa_alloc_num_free(const pa_alloc* a) { return a ? (int)a->free_list.size() : -1; }

int pa_alloc_ref(const pa_alloc* a, int block_id) {
  if (a == nullptr || block_id < 0 || block_id >= a->num_blocks) return -1;
  return a->ref[block_id];
}

int pa_alloc_num_seqs(const pa_alloc* a) { return a ? (int)a->seqs.size() : -1; }

int pa_slot_mapping(const int32_t* table, int num_rows, int max_blocks_per_seq, int block_size,
                    const int32_t* seq_idx, const int32_t* pos, int n, int64_t* slots_out) {
  if (n < 0 || block_size <= 0 || max_blocks_per_seq <= 0 || num_rows < 0) return PA_ERR_INVALID_ARG;
  if (n > 0 && (table == nullptr || seq_idx == nullptr || pos == nullptr || slots_out == nullptr))
    return PA_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const int s = seq_idx[i];
    const int p = pos[i];
    if (s < 0 || s >= num_rows || p < 0) return PA_ERR_INVALID_ARG;
    const int lb = p / block_size;
    if (lb >= max_blocks_per_seq) return PA_ERR_BAD_INDEX;
    const int32_t blk = table[(int64_t)s * max_blocks_per_seq + lb];
    if (blk < 0) return PA_ERR_BAD_INDEX;
    slots_out[i] = (int64_t)blk * block_size + p % block_size;
  }
  return PA_OK;
}

}  // extern "C"
