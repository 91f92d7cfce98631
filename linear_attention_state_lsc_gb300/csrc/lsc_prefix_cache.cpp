// lsc_prefix_cache.cpp -- the scheduler-side linear-state prefix cache of
// liblsc (host C++, no device code): one slot id space of free / live /
// checkpoint / reserved slots, a hash -> checkpoint table with pins and LRU
// reclaim, and the two-phase promotion (resolve reserves, commit hands off).
//
// Source: "Linear-State Prefix Cache 内部机制" (xLLM notes) §1-§7; the calls,
// their semantics and the readings of the page are stated in
// include/lsc_prefix_cache.h.
//
// Data structures, sized for tens of thousands of slots and resolve/commit on
// every scheduler step:
//   free slots    a bitmap; the lowest free id is a word scan + ctz
//   checkpoints   hash -> slot (an open-addressing table sized at creation, so
//                 no call after lsc_pc_create allocates for it) and per-slot
//                 hash; an intrusive
//                 doubly linked list in last-use order (head = least recent);
//                 reclaim walks it from the head past pinned entries
//   sequences     seq id -> (live slot, linear_state_initialized)
//   the step      the resolved rows' sequences, their pins and promotions
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "lsc_prefix_cache.h"

namespace {

// Open-addressing map from nonzero 64-bit keys to int32 values, linear probing,
// deletion by backward shift (no tombstones).  Capacity is a power of two set
// once; it must stay above the number of keys.
struct FlatMap {
  std::vector<uint64_t> keys;  // 0 = empty
  std::vector<int32_t> vals;
  uint64_t mask = 0;
  void init(size_t min_capacity) {
    size_t c = 16;
    while (c < min_capacity) c <<= 1;
    keys.assign(c, 0);
    vals.assign(c, 0);
    mask = c - 1;
  }
  // splitmix64 finaliser: spreads structured keys over the table
  static uint64_t mix(uint64_t x) {
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    return x ^ (x >> 31);
  }
  int32_t find(uint64_t k) const {
    for (uint64_t i = mix(k) & mask;; i = (i + 1) & mask) {
      if (keys[i] == k) return vals[i];
      if (keys[i] == 0) return -1;
    }
  }
  bool contains(uint64_t k) const { return find(k) >= 0; }
  void put(uint64_t k, int32_t v) {
    uint64_t i = mix(k) & mask;
    while (keys[i] != 0 && keys[i] != k) i = (i + 1) & mask;
    keys[i] = k;
    vals[i] = v;
  }
  void erase(uint64_t k) {
    uint64_t i = mix(k) & mask;
    while (keys[i] != k) {
      if (keys[i] == 0) return;
      i = (i + 1) & mask;
    }
    // backward shift: move later entries of the probe run into the hole
    for (uint64_t j = (i + 1) & mask; keys[j] != 0; j = (j + 1) & mask) {
      const uint64_t home = mix(keys[j]) & mask;
      // entry j may fill hole i when its home is not in (i, j] cyclically
      if (((j - home) & mask) >= ((j - i) & mask)) {
        keys[i] = keys[j];
        vals[i] = vals[j];
        i = j;
      }
    }
    keys[i] = 0;
  }
  void clear() { std::memset(keys.data(), 0, keys.size() * sizeof(uint64_t)); }
};

struct Promotion {
  lsc_prefix_hash hash;
  int64_t seq;
  int32_t live, replacement;
};

struct SeqInfo {
  int32_t slot;
  bool initialized;
};

}  // namespace

struct lsc_prefix_cache {
  int32_t num_slots = 0, block_size = 0;
  std::vector<uint8_t> state;     // LSC_SLOT_*
  std::vector<int32_t> pins;
  std::vector<lsc_prefix_hash> hash;
  std::vector<int32_t> prev, next;  // last-use list of checkpoints, -1 terminated
  int32_t lru_head = -1, lru_tail = -1;
  std::vector<uint64_t> free_bits;  // bit s set: slot s free
  FlatMap table;                  // hash -> checkpoint slot
  std::unordered_map<int64_t, SeqInfo> seqs;
  // the resolved step
  bool pending = false;
  std::vector<int64_t> step_seqs;
  std::vector<int32_t> step_pins;
  std::vector<Promotion> step_promotions;
  // scratch of resolve, kept to avoid reallocation
  FlatMap saving;                 // hashes promoted by this batch
  std::unordered_set<int64_t> seen;
};

namespace {

int32_t lowest_free(const lsc_prefix_cache *pc) {
  for (size_t w = 0; w < pc->free_bits.size(); ++w)
    if (pc->free_bits[w]) return (int32_t)(w * 64 + __builtin_ctzll(pc->free_bits[w]));
  return -1;
}
void set_free(lsc_prefix_cache *pc, int32_t s, bool f) {
  const uint64_t m = 1ull << (s % 64);
  if (f) pc->free_bits[s / 64] |= m;
  else pc->free_bits[s / 64] &= ~m;
}

void lru_unlink(lsc_prefix_cache *pc, int32_t s) {
  const int32_t p = pc->prev[s], n = pc->next[s];
  if (p >= 0) pc->next[p] = n;
  else pc->lru_head = n;
  if (n >= 0) pc->prev[n] = p;
  else pc->lru_tail = p;
  pc->prev[s] = pc->next[s] = -1;
}
void lru_push_recent(lsc_prefix_cache *pc, int32_t s) {
  pc->prev[s] = pc->lru_tail;
  pc->next[s] = -1;
  if (pc->lru_tail >= 0) pc->next[pc->lru_tail] = s;
  else pc->lru_head = s;
  pc->lru_tail = s;
}

// the least recently used checkpoint without pins, or -1
int32_t lru_victim(const lsc_prefix_cache *pc) {
  for (int32_t s = pc->lru_head; s >= 0; s = pc->next[s])
    if (pc->pins[s] == 0) return s;
  return -1;
}

void drop_checkpoint(lsc_prefix_cache *pc, int32_t s) {
  pc->table.erase(pc->hash[s]);
  pc->hash[s] = 0;
  lru_unlink(pc, s);
  pc->state[s] = LSC_SLOT_FREE;
  set_free(pc, s, true);
}

// [XN] §3.2 step 2 (insert_checkpoint): the slot joins the table as the most
// recently used entry
void insert_checkpoint(lsc_prefix_cache *pc, lsc_prefix_hash h, int32_t s) {
  pc->state[s] = LSC_SLOT_CHECKPOINT;
  pc->hash[s] = h;
  pc->table.put(h, s);
  lru_push_recent(pc, s);
}

bool can_promote(const lsc_prefix_cache *pc, int64_t tokens_after_step) {
  return tokens_after_step > 0 && tokens_after_step % pc->block_size == 0;
}

}  // namespace

extern "C" {

int lsc_pc_create(int32_t num_slots, int32_t block_size, lsc_prefix_cache **out) {
  if (!out || num_slots <= 0 || block_size <= 0) return LSC_ERR_INVALID_ARG;
  *out = nullptr;
  lsc_prefix_cache *pc = new (std::nothrow) lsc_prefix_cache();
  if (!pc) return LSC_ERR_NO_MEMORY;
  try {
    pc->num_slots = num_slots;
    pc->block_size = block_size;
    pc->state.assign(num_slots, LSC_SLOT_FREE);
    pc->pins.assign(num_slots, 0);
    pc->hash.assign(num_slots, 0);
    pc->prev.assign(num_slots, -1);
    pc->next.assign(num_slots, -1);
    pc->free_bits.assign((num_slots + 63) / 64, 0);
    for (int32_t s = 0; s < num_slots; ++s) set_free(pc, s, true);
    pc->table.init(2 * (size_t)num_slots);
  } catch (...) {
    delete pc;
    return LSC_ERR_NO_MEMORY;
  }
  *out = pc;
  return LSC_OK;
}

int lsc_pc_destroy(lsc_prefix_cache *pc) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  delete pc;
  return LSC_OK;
}

int lsc_pc_allocate_live_slot(lsc_prefix_cache *pc, int64_t seq_id, int32_t *slot) {
  if (!pc || !slot) return LSC_ERR_INVALID_ARG;
  if (pc->seqs.count(seq_id)) return LSC_ERR_INVALID_ARG;
  int32_t s = lowest_free(pc);
  const bool reclaim = s < 0;
  if (reclaim) {
    s = lru_victim(pc);
    if (s < 0) return LSC_ERR_NO_SLOT;
  }
  try {
    pc->seqs.emplace(seq_id, SeqInfo{s, false});
  } catch (...) {
    return LSC_ERR_NO_MEMORY;
  }
  if (reclaim) drop_checkpoint(pc, s);  // its hash leaves the table
  set_free(pc, s, false);
  pc->state[s] = LSC_SLOT_LIVE;
  *slot = s;
  return LSC_OK;
}

int lsc_pc_release_sequence(lsc_prefix_cache *pc, int64_t seq_id) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  auto it = pc->seqs.find(seq_id);
  if (it == pc->seqs.end()) return LSC_ERR_INVALID_ARG;
  if (pc->pending)  // the step's forward is writing this sequence's slot
    for (int64_t q : pc->step_seqs)
      if (q == seq_id) return LSC_ERR_ORDER;
  const int32_t s = it->second.slot;
  pc->seqs.erase(it);
  pc->state[s] = LSC_SLOT_FREE;
  set_free(pc, s, true);
  return LSC_OK;
}

int lsc_pc_match(lsc_prefix_cache *pc, lsc_prefix_hash h, int32_t *slot) {
  if (!pc || !slot) return LSC_ERR_INVALID_ARG;
  *slot = -1;
  if (h == 0) return LSC_OK;
  const int32_t s = pc->table.find(h);
  if (s < 0) return LSC_OK;
  ++pc->pins[s];
  lru_unlink(pc, s);
  lru_push_recent(pc, s);
  *slot = s;
  return LSC_OK;
}

int lsc_pc_unpin(lsc_prefix_cache *pc, int32_t slot) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  if (slot < 0 || slot >= pc->num_slots) return LSC_ERR_OUT_OF_RANGE;
  if (pc->state[slot] != LSC_SLOT_CHECKPOINT || pc->pins[slot] == 0) return LSC_ERR_INVALID_ARG;
  --pc->pins[slot];
  return LSC_OK;
}

int lsc_pc_resolve(lsc_prefix_cache *pc, const lsc_pc_row *rows, int32_t n, LinearStateCacheOp *ops,
                   uint8_t *linear_state_initialized, lsc_pc_report *report) {
  if (!pc || n < 0 || (n > 0 && (!rows || !ops))) return LSC_ERR_INVALID_ARG;
  if (pc->pending) return LSC_ERR_ORDER;
  // validate everything before changing anything
  try {
    pc->seen.clear();
    for (int32_t r = 0; r < n; ++r)
      if (!pc->seqs.count(rows[r].seq_id) || !pc->seen.insert(rows[r].seq_id).second) return LSC_ERR_INVALID_ARG;
    pc->step_seqs.clear();
    pc->step_pins.clear();
    pc->step_promotions.clear();
    if (pc->saving.keys.size() < 2 * (size_t)n) pc->saving.init(2 * (size_t)n);
    else pc->saving.clear();
    pc->step_seqs.reserve(n);
    pc->step_pins.reserve(n);
    pc->step_promotions.reserve(n);
  } catch (...) {
    return LSC_ERR_NO_MEMORY;
  }
  lsc_pc_report rep{};
  for (int32_t r = 0; r < n; ++r) {
    const lsc_pc_row &row = rows[r];
    const SeqInfo &si = pc->seqs.find(row.seq_id)->second;
    LinearStateCacheOp op{};
    op.linear_state_id = si.slot;
    op.restore_prefix_hash = row.restore_prefix_hash;
    op.save_prefix_hash = row.save_prefix_hash;
    op.restore_src_slot_id = -1;
    op.save_dst_slot_id = -1;
    op.reserved = 0;
    if (row.restore_prefix_hash != 0) {
      int32_t src = -1;
      lsc_pc_match(pc, row.restore_prefix_hash, &src);
      if (src >= 0) {
        pc->step_pins.push_back(src);
        ++rep.restore_hit;
      } else {
        ++rep.restore_miss;
      }
      op.restore_src_slot_id = src;
    }
    if (row.save_prefix_hash != 0) {
      if (pc->saving.contains(row.save_prefix_hash)) {
        ++rep.skip_duplicate;
      } else if (pc->table.contains(row.save_prefix_hash)) {
        ++rep.skip_cached;
      } else if (!can_promote(pc, row.tokens_after_step)) {
        ++rep.skip_unaligned;
      } else {
        const int32_t rs = lowest_free(pc);
        if (rs < 0) {
          ++rep.skip_no_slot;
        } else {
          set_free(pc, rs, false);
          pc->state[rs] = LSC_SLOT_RESERVED;
          pc->step_promotions.push_back(Promotion{row.save_prefix_hash, row.seq_id, si.slot, rs});
          pc->saving.put(row.save_prefix_hash, 1);
          op.save_dst_slot_id = si.slot;
          ++rep.save;
        }
      }
    }
    pc->step_seqs.push_back(row.seq_id);
    ops[r] = op;
    if (linear_state_initialized) linear_state_initialized[r] = si.initialized ? 1 : 0;
  }
  pc->pending = true;
  if (report) *report = rep;
  return LSC_OK;
}

int lsc_pc_commit(lsc_prefix_cache *pc) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  if (!pc->pending) return LSC_ERR_ORDER;
  // the forward wrote every resolved row's live slot ([XN] §5)
  for (int64_t seq : pc->step_seqs) pc->seqs.find(seq)->second.initialized = true;
  for (const Promotion &pr : pc->step_promotions) {
    // [XN] §3.2: move the live slot out of the sequence without freeing it,
    // make it the checkpoint of the hash, hand the sequence its replacement, cold
    insert_checkpoint(pc, pr.hash, pr.live);
    pc->state[pr.replacement] = LSC_SLOT_LIVE;
    SeqInfo &si = pc->seqs.find(pr.seq)->second;
    si.slot = pr.replacement;
    si.initialized = false;
  }
  for (int32_t s : pc->step_pins) --pc->pins[s];
  pc->step_seqs.clear();
  pc->step_pins.clear();
  pc->step_promotions.clear();
  pc->pending = false;
  return LSC_OK;
}

int lsc_pc_slot(const lsc_prefix_cache *pc, int32_t slot, int32_t *state, int32_t *pins, lsc_prefix_hash *h) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  if (slot < 0 || slot >= pc->num_slots) return LSC_ERR_OUT_OF_RANGE;
  if (state) *state = pc->state[slot];
  if (pins) *pins = pc->pins[slot];
  if (h) *h = pc->state[slot] == LSC_SLOT_CHECKPOINT ? pc->hash[slot] : 0;
  return LSC_OK;
}

int lsc_pc_sequence(const lsc_prefix_cache *pc, int64_t seq_id, int32_t *slot, int32_t *initialized) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  auto it = pc->seqs.find(seq_id);
  if (it == pc->seqs.end()) return LSC_ERR_INVALID_ARG;
  if (slot) *slot = it->second.slot;
  if (initialized) *initialized = it->second.initialized ? 1 : 0;
  return LSC_OK;
}

int lsc_pc_counts(const lsc_prefix_cache *pc, int32_t *n_free, int32_t *n_live, int32_t *n_checkpoint,
                  int32_t *n_reserved) {
  if (!pc) return LSC_ERR_INVALID_ARG;
  int32_t c[4] = {0, 0, 0, 0};
  for (uint8_t st : pc->state) ++c[st];
  if (n_free) *n_free = c[LSC_SLOT_FREE];
  if (n_live) *n_live = c[LSC_SLOT_LIVE];
  if (n_checkpoint) *n_checkpoint = c[LSC_SLOT_CHECKPOINT];
  if (n_reserved) *n_reserved = c[LSC_SLOT_RESERVED];
  return LSC_OK;
}

}  // extern "C"
