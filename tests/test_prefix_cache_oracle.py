"""Pins for the prefix-cache oracle (oracle/prefix_cache.py): the page's worked
promotion example (tests/golden/promotion_handoff.txt), each resolve skip rule
of §3.3 in isolation, the cold/warm bit of §5, pin protection, LRU reclaim order,
and the id-space invariants of §1-§2 under random operation sequences.

Source: xLLM notes "Linear-State Prefix Cache 内部机制".  CPU only.
"""
import random

import pytest

from oracle.prefix_cache import CHECKPOINT, LIVE, RESERVED, PrefixCache, PrefixCacheError

from _util import golden_kv


def filled(num_slots, n_live, block=16):
    """A cache whose slots 0..n_live-1 are held live by sequences 100 + i."""
    pc = PrefixCache(num_slots, block)
    for i in range(n_live):
        assert pc.allocate_live_slot(100 + i) == i
    return pc


def test_promotion_handoff_worked_example():
    """§3.1-§3.2: slot 7 promoted, replacement 9, sequence ends on 9 and cold."""
    g = golden_kv("promotion_handoff.txt")
    pc = filled(g["num_slots"], g["num_slots"] - 1)   # slots 0..8 live, 9 free
    seq = 100 + g["live_slot_before"]
    H = 0x5EED
    ops, init, rep = pc.resolve([(seq, 0, H, 32)])
    assert ops[0]["linear_state_id"] == g["op_linear_state_id"]
    assert ops[0]["save_dst_slot_id"] == g["op_save_dst_slot_id"]
    assert pc.slot(g["replacement_slot"])[0] == RESERVED
    assert pc.seq_slot[seq] == g["live_slot_before"]   # the sequence is not touched at resolve
    pc.commit()
    assert pc.seq_slot[seq] == g["sequence_slot_after"]
    assert int(pc.seq_initialized[seq]) == g["sequence_initialized_after"]
    st, pins, h = pc.slot(g["checkpoint_slot_after"])
    assert (st, h) == (CHECKPOINT, H)
    assert pc.match(H) == g["match_after"]


def test_skip_duplicate_hash_in_batch():
    """§3.3: several rows saving the same hash promote once."""
    pc = PrefixCache(8, 16)
    a, b = pc.allocate_live_slot(1), pc.allocate_live_slot(2)
    ops, _, rep = pc.resolve([(1, 0, 77, 16), (2, 0, 77, 16)])
    assert [o["save_dst_slot_id"] for o in ops] == [a, -1]
    assert rep["save"] == 1 and rep["skip_duplicate"] == 1
    pc.commit()
    assert pc.match(77) == a and pc.seq_slot[2] == b


def test_skip_already_cached():
    """§3.3: a prefix that already has a committed checkpoint is not saved again."""
    pc = PrefixCache(8, 16)
    pc.allocate_live_slot(1)
    pc.resolve([(1, 0, 5, 16)])
    pc.commit()
    before = pc.counts()
    ops, _, rep = pc.resolve([(1, 0, 5, 32)])
    assert ops[0]["save_dst_slot_id"] == -1 and rep["skip_cached"] == 1
    assert pc.counts() == before


def test_skip_cannot_promote_unaligned():
    """§3.1 + §3.3: only a block-aligned state is frozen; otherwise can_promote fails."""
    pc = PrefixCache(8, 16)
    pc.allocate_live_slot(1)
    for tokens in (0, 15, 17, 33):
        ops, _, rep = pc.resolve([(1, 0, 9, tokens)])
        assert ops[0]["save_dst_slot_id"] == -1 and rep["skip_unaligned"] == 1
        pc.commit()
    assert pc.counts() == (7, 1, 0, 0)


def test_skip_no_replacement_keeps_cache():
    """§3.3: with no free replacement the save is skipped; no checkpoint is evicted."""
    pc = PrefixCache(4, 16)
    pc.allocate_live_slot(1)
    pc.resolve([(1, 0, 11, 16)])
    pc.commit()                                   # slot 0 checkpoint 11, seq 1 on slot 1
    pc.allocate_live_slot(2)
    pc.allocate_live_slot(3)                      # slots 2, 3 live: nothing free
    ops, _, rep = pc.resolve([(2, 0, 12, 16)])
    assert ops[0]["save_dst_slot_id"] == -1 and rep["skip_no_slot"] == 1
    pc.commit()
    assert pc.slot(0) == (CHECKPOINT, 0, 11)


def test_hash_zero_means_not_requested():
    """§6.1: a zero hash requests nothing."""
    pc = PrefixCache(4, 16)
    pc.allocate_live_slot(1)
    ops, init, rep = pc.resolve([(1, 0, 0, 16)])
    assert ops[0]["restore_src_slot_id"] == -1 and ops[0]["save_dst_slot_id"] == -1
    assert rep == {k: 0 for k in rep}
    pc.commit()


def test_restore_hit_pins_until_commit():
    """§1 + §4: a match pins the checkpoint; a pinned checkpoint is not reclaimed."""
    pc = PrefixCache(3, 16)
    pc.allocate_live_slot(1)
    pc.resolve([(1, 0, 21, 16)])
    pc.commit()                                   # slot 0: checkpoint 21; seq 1 on slot 1
    pc.allocate_live_slot(2)                      # slot 2
    ops, _, rep = pc.resolve([(2, 21, 0, 16)])
    assert ops[0]["restore_src_slot_id"] == 0 and rep["restore_hit"] == 1
    assert pc.slot(0)[1] == 1
    with pytest.raises(PrefixCacheError):         # the only reclaimable slot is pinned
        pc.allocate_live_slot(3)
    pc.commit()
    assert pc.slot(0)[1] == 0
    assert pc.allocate_live_slot(3) == 0          # unpinned now: reclaimed
    assert pc.match(21) == -1


def test_restore_miss():
    pc = PrefixCache(4, 16)
    pc.allocate_live_slot(1)
    ops, _, rep = pc.resolve([(1, 99, 0, 16)])
    assert ops[0]["restore_src_slot_id"] == -1 and rep["restore_miss"] == 1
    pc.commit()


def test_initialized_follows_the_slot():
    """§5: cold on allocation, warm once a forward wrote the slot, cold again
    after a promotion hands the sequence a fresh slot."""
    pc = PrefixCache(8, 16)
    pc.allocate_live_slot(1)
    _, init, _ = pc.resolve([(1, 0, 0, 8)])
    assert init == [0]
    pc.commit()
    _, init, _ = pc.resolve([(1, 0, 3, 16)])
    assert init == [1]
    pc.commit()
    assert pc.seq_initialized[1] is False
    _, init, _ = pc.resolve([(1, 0, 0, 17)])
    assert init == [0]
    pc.commit()
    assert pc.seq_initialized[1] is True


def test_lru_reclaim_order():
    """§1: unpinned checkpoints are reclaimed least recently used first; a match
    refreshes a checkpoint."""
    pc = PrefixCache(4, 16)
    for seq, h in ((1, 31), (2, 32), (3, 33)):
        pc.allocate_live_slot(seq)
        pc.resolve([(seq, 0, h, 16)])
        pc.commit()
        pc.release_sequence(seq)
    # three checkpoints, inserted 31, 32, 33; touch 31 again
    s31 = pc.match(31)
    pc.unpin(s31)
    pc.allocate_live_slot(10)                     # takes the one free slot
    victim = pc.slot_of_hash[32]
    assert pc.allocate_live_slot(11) == victim    # 32 is now the least recent
    assert pc.match(32) == -1 and pc.match(31) >= 0


def test_errors_leave_state_unchanged():
    pc = PrefixCache(4, 16)
    pc.allocate_live_slot(1)
    with pytest.raises(PrefixCacheError):
        pc.resolve([(1, 0, 0, 16), (1, 0, 0, 16)])    # same sequence twice
    with pytest.raises(PrefixCacheError):
        pc.resolve([(2, 0, 0, 16)])                   # unknown sequence
    with pytest.raises(PrefixCacheError):
        pc.commit()                                   # nothing resolved
    with pytest.raises(PrefixCacheError):
        pc.allocate_live_slot(1)                      # already holds a slot
    assert pc.counts() == (3, 1, 0, 0) and pc.pending is None
    pc.resolve([(1, 0, 0, 16)])
    with pytest.raises(PrefixCacheError):
        pc.release_sequence(1)                        # its forward is writing the slot
    with pytest.raises(PrefixCacheError):
        pc.resolve([(1, 0, 0, 16)])                   # previous step not committed
    pc.commit()
    pc.release_sequence(1)
    assert pc.counts() == (4, 0, 0, 0)


def check_invariants(pc):
    """§1-§2: one id space, each slot in exactly one state; a checkpoint belongs
    to exactly one hash; sequences hold distinct live slots."""
    assert sum(pc.counts()) == pc.num_slots
    ck = [s for s in range(pc.num_slots) if pc.state[s] == CHECKPOINT]
    assert sorted(pc.hash_of_slot) == ck
    assert {pc.slot_of_hash[h] for h in pc.slot_of_hash} == set(ck)
    assert all(pc.hash_of_slot[pc.slot_of_hash[h]] == h for h in pc.slot_of_hash)
    live = sorted(pc.seq_slot.values())
    assert len(set(live)) == len(live)
    assert live == [s for s in range(pc.num_slots) if pc.state[s] == LIVE]
    assert all(pc.pins[s] == 0 for s in range(pc.num_slots) if pc.state[s] != CHECKPOINT)
    assert all(p >= 0 for p in pc.pins)


@pytest.mark.parametrize("seed", range(6))
def test_random_steps_keep_invariants(seed):
    rng = random.Random(seed)
    pc = PrefixCache(12, 4)
    next_seq = 0
    hashes = [0] + list(range(1, 9))
    for _ in range(300):
        r = rng.random()
        if r < 0.25:
            try:
                pc.allocate_live_slot(next_seq)
                next_seq += 1
            except PrefixCacheError:
                pass
        elif r < 0.35 and pc.seq_slot:
            pc.release_sequence(rng.choice(sorted(pc.seq_slot)))
        elif pc.seq_slot:
            seqs = rng.sample(sorted(pc.seq_slot), rng.randint(1, len(pc.seq_slot)))
            rows = [(s, rng.choice(hashes), rng.choice(hashes), rng.randint(0, 12)) for s in seqs]
            pins_before = sum(pc.pins)
            ops, init, rep = pc.resolve(rows)
            assert sum(pc.pins) == pins_before + rep["restore_hit"]
            for o, (s, rh, sh, t) in zip(ops, rows):
                assert o["linear_state_id"] == pc.seq_slot[s]
                if o["restore_src_slot_id"] >= 0:
                    assert pc.state[o["restore_src_slot_id"]] == CHECKPOINT
            pc.commit()
            assert sum(pc.pins) == pins_before
        check_invariants(pc)
