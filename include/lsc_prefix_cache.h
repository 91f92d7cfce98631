/*
 * lsc_prefix_cache.h -- C ABI of the scheduler-side linear-state prefix cache
 * of liblsc: the slot id space, the checkpoint table and the two-phase
 * promotion that produce the LinearStateCacheOp rows lsc_restore consumes.
 * Host memory only; no call touches a GPU.
 *
 * Source, cited by page title and section:
 *   [XN] "Linear-State Prefix Cache 内部机制" (xLLM notes)
 *
 * Model ([XN] §1-§2): one id space [0, num_slots) shared by
 *   free        not held by anyone;
 *   live        held by one sequence, overwritten in place by every forward;
 *   checkpoint  a frozen state in the table under its prefix hash, restorable,
 *               reclaimed least recently used first when not pinned;
 *   reserved    a free slot set aside by resolve as a promotion's replacement.
 * These slot ids are the pool's slot ids (lsc_pool_create's num_slots).
 *
 * One step ([XN] §3.1, §7): the caller builds one lsc_pc_row per batch row
 * (sequence, restore hash, save hash: the BUILD stage), calls lsc_pc_resolve
 * before the forward (it fills the LinearStateCacheOp rows and the
 * linear_state_initialized bits for lsc_restore), runs the forward, then calls
 * lsc_pc_commit, which performs the promotions ([XN] §3.2).
 *
 * Readings of the page (it leaves these open):
 *   - can_promote: a promotion freezes the block-aligned state of this step
 *     ([XN] §3.1), so a row is promotable only when tokens_after_step is a
 *     positive multiple of the cache's block_size.
 *   - Free slots are handed out lowest id first.  lsc_pc_allocate_live_slot
 *     reclaims the least recently used unpinned checkpoint when no slot is
 *     free; a replacement slot at resolve never reclaims ([XN] §3.3).
 *   - "Recently used" advances on every match hit and every insertion.
 *   - resolve's matches pin their checkpoints until the step's commit, since
 *     the restore copy that reads them runs during the forward.
 *
 * Conventions: the return codes of lsc.h; on an error return nothing changed.
 * A cache is not thread-safe: one thread (the scheduler) drives it.
 */
#ifndef LSC_PREFIX_CACHE_H
#define LSC_PREFIX_CACHE_H

#include "lsc.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lsc_prefix_cache lsc_prefix_cache;

/* Slot states reported by lsc_pc_slot. */
#define LSC_SLOT_FREE 0
#define LSC_SLOT_LIVE 1
#define LSC_SLOT_CHECKPOINT 2
#define LSC_SLOT_RESERVED 3

/* One batch row of a step, as the BUILD stage knows it ([XN] §7 stage 1). */
typedef struct {
  int64_t seq_id;                      /* a sequence holding a live slot */
  lsc_prefix_hash restore_prefix_hash; /* nonzero: restore requested ([XN] §6.1) */
  lsc_prefix_hash save_prefix_hash;    /* nonzero: save requested */
  int64_t tokens_after_step;           /* tokens the sequence has computed once this step's forward is done */
} lsc_pc_row;

/* Counts of one lsc_pc_resolve call ([XN] §3.3 names the four skips). */
typedef struct {
  int32_t restore_hit, restore_miss;
  int32_t save;              /* promotions reserved */
  int32_t skip_duplicate;    /* another row of the batch saves the same hash */
  int32_t skip_cached;       /* the hash already has a committed checkpoint */
  int32_t skip_unaligned;    /* can_promote failed: tokens_after_step not block-aligned */
  int32_t skip_no_slot;      /* no free replacement slot (nothing is evicted for it) */
  int32_t reserved;
} lsc_pc_report;

/* Create a cache over slot ids [0, num_slots), all free.  block_size > 0 is the
 * KV block size of the promotion rule.  Errors: INVALID_ARG, NO_MEMORY. */
int lsc_pc_create(int32_t num_slots, int32_t block_size, lsc_prefix_cache **out);
int lsc_pc_destroy(lsc_prefix_cache *pc);

/* Give sequence seq_id an empty live slot ([XN] §1 allocate_live_slot): the
 * lowest free id, else the least recently used unpinned checkpoint, whose hash
 * leaves the table.  The sequence starts cold (linear_state_initialized = 0,
 * [XN] §5).  Errors: INVALID_ARG (the sequence already holds a slot),
 * NO_SLOT (nothing free or reclaimable). */
int lsc_pc_allocate_live_slot(lsc_prefix_cache *pc, int64_t seq_id, int32_t *slot);

/* A finished sequence returns its live slot to the free list.  Errors:
 * INVALID_ARG (unknown sequence), ORDER (the sequence is a row of the resolved
 * step, whose forward writes its slot: release it after lsc_pc_commit). */
int lsc_pc_release_sequence(lsc_prefix_cache *pc, int64_t seq_id);

/* Look up a prefix hash ([XN] §1, §4).  On a hit *slot is the checkpoint slot,
 * which is pinned (not reclaimable) until lsc_pc_unpin, and becomes the most
 * recently used; on a miss (or hash 0) *slot = -1 and nothing changes. */
int lsc_pc_match(lsc_prefix_cache *pc, lsc_prefix_hash hash, int32_t *slot);
/* Release one pin taken by lsc_pc_match.  Errors: OUT_OF_RANGE, INVALID_ARG
 * (the slot is not a pinned checkpoint). */
int lsc_pc_unpin(lsc_prefix_cache *pc, int32_t slot);

/* RESOLVE ([XN] §3.1, §3.3, §6, §7 stage 2), before the forward.  For each row
 * in order:
 *   ops[r].linear_state_id     = the sequence's live slot
 *   ops[r].restore_src_slot_id = match(restore hash), -1 on a miss or hash 0;
 *                                a hit stays pinned until lsc_pc_commit
 *   ops[r].save_dst_slot_id    = the live slot when a promotion is reserved,
 *                                else -1: skipped when another row already
 *                                saves the hash, the hash is cached, the row is
 *                                not block-aligned, or no slot is free (in that
 *                                order); a reservation takes the lowest free
 *                                slot as the replacement
 *   ops[r] hashes              = the row's hashes, reserved = 0
 *   linear_state_initialized[r] = the sequence's cold/warm bit ([XN] §5)
 * ops (host [n]) and linear_state_initialized (host [n], may be NULL) are
 * written; report may be NULL.  Errors: INVALID_ARG (unknown or repeated
 * sequence, n < 0, NULL arrays with n > 0), ORDER (the previous step is not
 * committed). */
int lsc_pc_resolve(lsc_prefix_cache *pc, const lsc_pc_row *rows, int32_t n, LinearStateCacheOp *ops,
                   uint8_t *linear_state_initialized, lsc_pc_report *report);

/* COMMIT ([XN] §3.2, §5, §7 stage 4), after the forward wrote the live slots:
 * every sequence of the resolved batch becomes warm; then, per reserved
 * promotion in row order, the old live slot becomes the checkpoint of its
 * hash (moved out of the sequence, not freed), and the sequence takes the
 * replacement slot, cold.  Finally the step's match pins are released.
 * Errors: ORDER (nothing resolved). */
int lsc_pc_commit(lsc_prefix_cache *pc);

/* Introspection.  lsc_pc_slot: state (LSC_SLOT_*), pin count and checkpoint
 * hash (0 unless a checkpoint) of one slot; any out pointer may be NULL.
 * lsc_pc_sequence: the live slot and cold/warm bit of a sequence.
 * lsc_pc_counts: slots per state. */
int lsc_pc_slot(const lsc_prefix_cache *pc, int32_t slot, int32_t *state, int32_t *pins, lsc_prefix_hash *hash);
int lsc_pc_sequence(const lsc_prefix_cache *pc, int64_t seq_id, int32_t *slot, int32_t *initialized);
int lsc_pc_counts(const lsc_prefix_cache *pc, int32_t *n_free, int32_t *n_live, int32_t *n_checkpoint,
                  int32_t *n_reserved);

#ifdef __cplusplus
}
#endif

#endif /* LSC_PREFIX_CACHE_H */
