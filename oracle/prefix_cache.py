"""Plain model of the scheduler-side linear-state prefix cache.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/ and bench.py's CPU legs
import this module.  It is written for reading, not speed: lists, dicts and
linear scans, one method per operation the page names.

Source: "Linear-State Prefix Cache 内部机制" (xLLM notes).
  §1-§2  One id space [0, num_slots) holds free, live and checkpoint slots; a
         slot's state is told apart by its owner and its pin count.
  §1     match(hash) on a hit pins the checkpoint; unpinned checkpoints are
         reclaimed least recently used first.
  §3.1   resolve (before forward) only reserves promotions; commit (after
         forward) performs them.
  §3.2   The hand-off: the live slot is moved out of the sequence without being
         freed, inserted as the checkpoint of the hash, and the sequence takes
         the replacement slot reserved at resolve, marked cold.
  §3.3   resolve skips a save whose hash another row of the batch already
         saves, whose hash is already cached, whose row cannot be promoted, or
         for which no free replacement slot exists (no eviction for this).
  §4     restore_src_slot_id is the slot match() found, -1 on a miss.
  §5     linear_state_initialized follows the slot: valid after a forward
         wrote it, cold again after promotion hands over a fresh slot.
  §6     LinearStateCacheOp: linear_state_id, restore hash and source slot,
         save hash and save_dst_slot_id (the old live slot when a promotion
         really happens, -1 otherwise).

Readings where the page is silent (also listed in the design notes):
  * can_promote: the state frozen by a promotion is the one at a block-aligned
    boundary (§3.1), so a row can be promoted only when the tokens it has
    computed once this step's forward is done are a positive multiple of
    block_size.
  * Free slots are handed out lowest id first; a live-slot allocation with no
    free slot reclaims the least recently used unpinned checkpoint (§1 "LRU 可回收").
    A replacement slot at resolve never reclaims (§3.3).
  * "Recently used" is a logical clock advanced by every match hit and insert.
  * Pins taken by resolve's matches are released by the step's commit: the
    restore copy that reads the checkpoint runs during the forward.
  * Each sequence appears at most once per batch; resolve may not run again
    before commit, and a sequence of the resolved step may not be released
    before the commit (its forward is writing the live slot).
"""

FREE, LIVE, CHECKPOINT, RESERVED = 0, 1, 2, 3


class PrefixCacheError(Exception):
    """kind: "arg" (bad argument), "no_slot" (nothing free or reclaimable) or
    "order" (a call out of step order)."""

    def __init__(self, what, kind="arg"):
        super().__init__(what)
        self.kind = kind


class PrefixCache:
    def __init__(self, num_slots, block_size):
        if num_slots <= 0 or block_size <= 0:
            raise PrefixCacheError("bad size")
        self.num_slots = num_slots
        self.block_size = block_size
        self.state = [FREE] * num_slots
        self.pins = [0] * num_slots
        self.hash_of_slot = {}      # checkpoint slot -> hash
        self.slot_of_hash = {}      # hash -> checkpoint slot
        self.last_use = {}          # checkpoint slot -> clock value
        self.clock = 0
        self.seq_slot = {}          # sequence -> live slot
        self.seq_initialized = {}   # sequence -> linear_state_initialized
        self.pending = None         # the resolved step awaiting commit

    # -- the id space ------------------------------------------------------
    def _lowest_free(self):
        for s in range(self.num_slots):
            if self.state[s] == FREE:
                return s
        return None

    def _lru_unpinned_checkpoint(self):
        best = None
        for s in range(self.num_slots):
            if self.state[s] == CHECKPOINT and self.pins[s] == 0:
                if best is None or self.last_use[s] < self.last_use[best]:
                    best = s
        return best

    def _drop_checkpoint(self, s):
        h = self.hash_of_slot.pop(s)
        del self.slot_of_hash[h]
        del self.last_use[s]
        self.state[s] = FREE

    def _touch(self, s):
        self.clock += 1
        self.last_use[s] = self.clock

    # -- sequences ---------------------------------------------------------
    def allocate_live_slot(self, seq):
        if seq in self.seq_slot:
            raise PrefixCacheError("sequence already holds a slot")
        s = self._lowest_free()
        if s is None:
            s = self._lru_unpinned_checkpoint()
            if s is None:
                raise PrefixCacheError("no slot", "no_slot")
            self._drop_checkpoint(s)
        self.state[s] = LIVE
        self.seq_slot[seq] = s
        self.seq_initialized[seq] = False
        return s

    def release_sequence(self, seq):
        if seq not in self.seq_slot:
            raise PrefixCacheError("unknown sequence")
        if self.pending is not None and seq in self.pending["seqs"]:
            raise PrefixCacheError("the sequence is in the resolved step", "order")
        s = self.seq_slot.pop(seq)
        del self.seq_initialized[seq]
        self.state[s] = FREE

    # -- the checkpoint table ----------------------------------------------
    def match(self, h):
        if h == 0 or h not in self.slot_of_hash:
            return -1
        s = self.slot_of_hash[h]
        self.pins[s] += 1
        self._touch(s)
        return s

    def unpin(self, s):
        if not (0 <= s < self.num_slots) or self.state[s] != CHECKPOINT or self.pins[s] == 0:
            raise PrefixCacheError("not a pinned checkpoint")
        self.pins[s] -= 1

    def insert_checkpoint(self, h, s):
        self.state[s] = CHECKPOINT
        self.hash_of_slot[s] = h
        self.slot_of_hash[h] = s
        self._touch(s)

    # -- one step ----------------------------------------------------------
    def can_promote(self, tokens_after_step):
        return tokens_after_step > 0 and tokens_after_step % self.block_size == 0

    def resolve(self, rows):
        """rows: list of (seq, restore_hash, save_hash, tokens_after_step).
        Returns (ops, initialized, report); ops are dicts with the six
        LinearStateCacheOp fields."""
        if self.pending is not None:
            raise PrefixCacheError("previous step not committed", "order")
        seen = set()
        for seq, _, _, _ in rows:
            if seq not in self.seq_slot or seq in seen:
                raise PrefixCacheError("bad row")
            seen.add(seq)
        report = {"restore_hit": 0, "restore_miss": 0, "save": 0, "skip_duplicate": 0,
                  "skip_cached": 0, "skip_unaligned": 0, "skip_no_slot": 0}
        ops, initialized, pins, promotions, saving = [], [], [], [], set()
        for seq, rh, sh, tokens in rows:
            live = self.seq_slot[seq]
            src = -1
            if rh != 0:
                src = self.match(rh)
                if src >= 0:
                    pins.append(src)
                    report["restore_hit"] += 1
                else:
                    report["restore_miss"] += 1
            dst = -1
            if sh != 0:
                if sh in saving:
                    report["skip_duplicate"] += 1
                elif sh in self.slot_of_hash:
                    report["skip_cached"] += 1
                elif not self.can_promote(tokens):
                    report["skip_unaligned"] += 1
                else:
                    rep = self._lowest_free()
                    if rep is None:
                        report["skip_no_slot"] += 1
                    else:
                        self.state[rep] = RESERVED
                        promotions.append((sh, seq, live, rep))
                        saving.add(sh)
                        dst = live
                        report["save"] += 1
            ops.append({"linear_state_id": live, "restore_src_slot_id": src,
                        "restore_prefix_hash": rh, "save_prefix_hash": sh,
                        "save_dst_slot_id": dst, "reserved": 0})
            initialized.append(1 if self.seq_initialized[seq] else 0)
        self.pending = {"seqs": [r[0] for r in rows], "pins": pins, "promotions": promotions}
        return ops, initialized, report

    def commit(self):
        if self.pending is None:
            raise PrefixCacheError("nothing to commit", "order")
        # the forward wrote every row's live slot
        for seq in self.pending["seqs"]:
            self.seq_initialized[seq] = True
        for h, seq, live, rep in self.pending["promotions"]:
            # move the live slot out of the sequence without freeing it ...
            # ... make it the checkpoint of h ...
            self.insert_checkpoint(h, live)
            # ... and hand the sequence its replacement, cold
            self.state[rep] = LIVE
            self.seq_slot[seq] = rep
            self.seq_initialized[seq] = False
        for s in self.pending["pins"]:
            self.pins[s] -= 1
        self.pending = None

    # -- introspection -----------------------------------------------------
    def slot(self, s):
        return self.state[s], self.pins[s], self.hash_of_slot.get(s, 0)

    def counts(self):
        return tuple(sum(1 for x in self.state if x == k) for k in (FREE, LIVE, CHECKPOINT, RESERVED))
