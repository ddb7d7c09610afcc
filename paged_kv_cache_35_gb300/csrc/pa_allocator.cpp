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
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"

// Prefix cache ([cb] "Prefix 캐싱" and "제거" sections of the continuous
// batching page): every completed block of a sequence whose token ids are
// known is keyed by its whole prefix (the token ids from position 0 to the
// end of the block).  A later sequence whose prompt starts with the same
// prefix reuses the block instead of recomputing it.  A block whose last
// reference goes away keeps its content and key ("initialized") and can still
// be matched; when no uninitialized block is left, the most recently freed
// initialized block is demoted (its key dropped) and handed out.
//
// The prefix key is represented by a 128-bit chained fingerprint of the
// token ids plus the block's own token ids, compared on every match.
struct PrefixKey {
  uint64_t a = 0, b = 0;
  bool operator==(const PrefixKey& o) const { return a == o.a && b == o.b; }
};
struct PrefixKeyHash {
  size_t operator()(const PrefixKey& k) const { return (size_t)(k.a ^ (k.b * 0x9e3779b97f4a7c15ULL)); }
};

struct pa_alloc {
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
    bool tracked = false;          // token ids known for every position
    std::vector<int32_t> tokens;   // ids of positions 0 .. len-1 (tracked only)
    std::vector<PrefixKey> keys;   // prefix key of each full block (tracked only)
  };
  int num_blocks = 0;
  int block_size = 0;
  bool prefix_cache = false;
  std::vector<int32_t> free_list;  // uninitialized free blocks, taken from the back
  std::vector<int32_t> ref;
  std::unordered_map<int, Seq> seqs;
  // prefix cache
  std::unordered_map<PrefixKey, int32_t, PrefixKeyHash> cache;
  std::vector<uint8_t> cached;                  // block holds a cache entry
  std::vector<PrefixKey> key;                   // its key
  std::vector<std::vector<int32_t>> block_ids;  // its own token ids
  std::list<int32_t> init_list;                 // initialized free blocks, oldest first
  std::vector<std::list<int32_t>::iterator> init_pos;

  int num_free() const { return (int)(free_list.size() + init_list.size()); }

  void uncache(int32_t b) {
    cache.erase(key[b]);
    cached[b] = 0;
    block_ids[b].clear();
  }
  int32_t take() {
    int32_t b;
    if (!free_list.empty()) {
      b = free_list.back();
      free_list.pop_back();
    } else {  // demote the most recently freed initialized block
      b = init_list.back();
      init_list.pop_back();
      uncache(b);
    }
    ref[b] = 1;
    return b;
  }
  bool release(int32_t b) {
    if (ref[b] <= 0) return false;
    if (--ref[b] == 0) {
      if (prefix_cache && cached[b]) {
        init_list.push_back(b);
        init_pos[b] = std::prev(init_list.end());
      } else {
        free_list.push_back(b);
      }
    }
    return true;
  }
  // a cached block gains a reference (taken back from the initialized list if free)
  void reuse(int32_t b) {
    if (ref[b] == 0) init_list.erase(init_pos[b]);
    ++ref[b];
  }
  static uint64_t mix64(uint64_t x) {
    x ^= x >> 33;
    x *= 0xff51afd7ed558ccdULL;
    x ^= x >> 33;
    x *= 0xc4ceb9fe1a85ec53ULL;
    x ^= x >> 33;
    return x;
  }
  // key of a block: the previous block's key chained with this block's ids
  PrefixKey next_key(const PrefixKey& prev, const int32_t* ids) const {
    uint64_t x = prev.a ^ 0x243f6a8885a308d3ULL, y = prev.b ^ 0x13198a2e03707344ULL;
    for (int i = 0; i < block_size; ++i) {
      const uint64_t t = (uint32_t)ids[i];
      x = mix64(x + t * 0x9e3779b97f4a7c15ULL + (uint64_t)i);
      y = mix64((y ^ (t << 17)) + 0xd6e8feb86659fd93ULL * (uint64_t)(i + 1));
    }
    return PrefixKey{x, y};
  }
  // the cached block for (key, ids), or -1
  int32_t lookup(const PrefixKey& k, const int32_t* ids) const {
    auto it = cache.find(k);
    if (it == cache.end()) return -1;
    const auto& own = block_ids[it->second];
    return std::equal(own.begin(), own.end(), ids) ? it->second : -1;
  }
  // a tracked sequence's last block just filled: give it a cache entry unless
  // its prefix already has one
  void publish(Seq& sq) {
    const int nfull = (int)(sq.len / block_size);
    const int32_t* ids = sq.tokens.data() + (int64_t)(nfull - 1) * block_size;
    const PrefixKey k = next_key(nfull > 1 ? sq.keys[nfull - 2] : PrefixKey{}, ids);
    sq.keys.push_back(k);
    if (cache.count(k)) return;
    const int32_t b = sq.blocks.back();
    cache.emplace(k, b);
    cached[b] = 1;
    key[b] = k;
    block_ids[b].assign(ids, ids + block_size);
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

int pa_alloc_create_ex(int num_blocks, int block_size, int flags, pa_alloc** out) {
  if (out == nullptr || num_blocks <= 0 || block_size <= 0 || (flags & ~PA_ALLOC_PREFIX_CACHE) != 0)
    return PA_ERR_INVALID_ARG;
  pa_alloc* a = new (std::nothrow) pa_alloc();
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->prefix_cache = (flags & PA_ALLOC_PREFIX_CACHE) != 0;
  a->free_list.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) a->free_list[i] = i;
  a->ref.assign(num_blocks, 0);
  if (a->prefix_cache) {
    a->cached.assign(num_blocks, 0);
    a->key.assign(num_blocks, PrefixKey{});
    a->block_ids.assign(num_blocks, std::vector<int32_t>());
    a->init_pos.assign(num_blocks, a->init_list.end());
  }
  *out = a;
  return PA_OK;
}

int pa_alloc_create(int num_blocks, int block_size, pa_alloc** out) {
  return pa_alloc_create_ex(num_blocks, block_size, 0, out);
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

}  // extern "C"

namespace {

int append_impl(pa_alloc* a, const int* seq_ids, const int32_t* token_ids, int n, int64_t* slots_out,
                int32_t* copy_pairs_out, int* n_pairs_out) {
  if (a == nullptr || n < 0 || (n > 0 && (seq_ids == nullptr || slots_out == nullptr))) return PA_ERR_INVALID_ARG;
  std::unordered_set<int> seen;
  for (int i = 0; i < n; ++i) {
    if (!a->seqs.count(seq_ids[i]) || !seen.insert(seq_ids[i]).second) return PA_ERR_INVALID_ARG;
  }
  if (blocks_needed(*a, seq_ids, n) > a->num_free()) return PA_ERR_NO_FREE_BLOCKS;
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
    if (sq.tracked) {
      if (token_ids == nullptr) {  // ids no longer known: the sequence leaves the cache
        sq.tracked = false;
        sq.tokens.clear();
        sq.keys.clear();
      } else {
        sq.tokens.push_back(token_ids[i]);
        if (a->prefix_cache && sq.len % B == 0) a->publish(sq);
      }
    }
  }
  if (n_pairs_out != nullptr) *n_pairs_out = np;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_alloc_append_slots(pa_alloc* a, const int* seq_ids, int n, int64_t* slots_out, int32_t* copy_pairs_out,
                          int* n_pairs_out) {
  return append_impl(a, seq_ids, nullptr, n, slots_out, copy_pairs_out, n_pairs_out);
}

int pa_alloc_append_tokens(pa_alloc* a, const int* seq_ids, const int32_t* token_ids, int n, int64_t* slots_out,
                           int32_t* copy_pairs_out, int* n_pairs_out) {
  if (n > 0 && token_ids == nullptr) return PA_ERR_INVALID_ARG;
  return append_impl(a, seq_ids, token_ids, n, slots_out, copy_pairs_out, n_pairs_out);
}

int pa_alloc_add_seq_prefix(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, int* n_reused_tokens) {
  if (a == nullptr || seq_id < 0 || a->seqs.count(seq_id) || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
    return PA_ERR_INVALID_ARG;
  pa_alloc::Seq sq;
  sq.tracked = true;
  const int B = a->block_size;
  if (a->prefix_cache) {
    PrefixKey k;
    for (int i = 0; (int64_t)(i + 1) * B <= n_tokens; ++i) {
      const int32_t* ids = tokens + (int64_t)i * B;
      k = a->next_key(k, ids);
      const int32_t b = a->lookup(k, ids);
      if (b < 0) break;
      a->reuse(b);
      sq.blocks.push_back(b);
      sq.keys.push_back(k);
      sq.tokens.insert(sq.tokens.end(), ids, ids + B);
      sq.len += B;
    }
  }
  if (n_reused_tokens != nullptr) *n_reused_tokens = (int)sq.len;
  a->seqs.emplace(seq_id, std::move(sq));
  return PA_OK;
}

int pa_alloc_prefix_stats(const pa_alloc* a, int* cached_blocks, int* initialized_free_blocks) {
  if (a == nullptr) return PA_ERR_INVALID_ARG;
  if (cached_blocks) *cached_blocks = (int)a->cache.size();
  if (initialized_free_blocks) *initialized_free_blocks = (int)a->init_list.size();
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

// Groups for pa_decode_grouped, from the tables: runs of consecutive listed
// sequences (at most max_group) whose tables start with the same blocks.  A
// run grows while the next sequence shares at least its first full block with
// the run's first sequence; the run's prefix is the leading blocks that every
// member holds in common with the first and has filled (length at least
// (b + 1) * block_size), in tokens, rounded down to a multiple of 16.  A run
// of one sequence has prefix 0.
int pa_alloc_prefix_groups(const pa_alloc* a, const int* seq_ids, int n, int max_group, int32_t* group_start_out,
                           int32_t* group_prefix_out, int* num_groups_out) {
  if (a == nullptr || n < 0 || max_group < 1 || max_group > 8 || num_groups_out == nullptr ||
      (n > 0 && (seq_ids == nullptr || group_prefix_out == nullptr)) || group_start_out == nullptr)
    return PA_ERR_INVALID_ARG;
  std::vector<const pa_alloc::Seq*> sq(n);
  for (int i = 0; i < n; ++i) {
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
    sq[i] = &it->second;
  }
  const int64_t B = a->block_size;
  auto full_blocks = [&](const pa_alloc::Seq& s) { return std::min<int64_t>(s.len / B, (int64_t)s.blocks.size()); };
  int G = 0;
  for (int i = 0; i < n;) {
    const pa_alloc::Seq& first = *sq[i];
    int64_t common = full_blocks(first);
    int j = i + 1;
    while (j < n && j - i < max_group && common > 0) {
      const pa_alloc::Seq& m = *sq[j];
      const int64_t lim = std::min(common, full_blocks(m));
      int64_t c = 0;
      while (c < lim && m.blocks[c] == first.blocks[c]) ++c;
      if (c == 0) break;
      common = c;
      ++j;
    }
    int64_t prefix = j - i > 1 ? common * B : 0;
    prefix = std::min<int64_t>(prefix, INT32_MAX) / 16 * 16;
    group_start_out[G] = i;
    group_prefix_out[G] = (int32_t)prefix;
    ++G;
    i = j;
  }
  group_start_out[G] = n;
  *num_groups_out = G;
  return PA_OK;
}

int pa_alloc_num_free(const pa_alloc* a) { return a ? a->num_free() : -1; }

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
