"""The library's prefix cache (include/lsc_prefix_cache.h) against the oracle
(oracle/prefix_cache.py): the same random operation sequences on both sides,
every output compared exactly -- return code class, ops rows, cold/warm bits,
resolve counts, and after every call the state, pins and hash of every slot and
the live slot and bit of every sequence.  Plus the page's worked example through
the C ABI.  Host code only: CPU tests.

Source: xLLM notes "Linear-State Prefix Cache 内部机制" §1-§7.
"""
import random

import numpy as np
import pytest

from oracle.prefix_cache import PrefixCache, PrefixCacheError
from linear_attention_state_lsc_gb300 import lsc as L

from _util import golden_kv

KIND_CODE = {"arg": L.LSC_ERR_INVALID_ARG, "no_slot": L.LSC_ERR_NO_SLOT, "order": L.LSC_ERR_ORDER}


@pytest.fixture
def lib_cache(lsc):
    made = []

    def make(num_slots, block):
        rc, pc = L.lsc_pc_create(num_slots, block)
        assert rc == L.LSC_OK
        made.append(pc)
        return pc
    yield make
    for pc in made:
        assert L.lsc_pc_destroy(pc) == L.LSC_OK


def same_state(pc, orc):
    for s in range(orc.num_slots):
        rc, st, pins, h = L.lsc_pc_slot(pc, s)
        assert rc == L.LSC_OK
        assert (st, pins, h) == orc.slot(s), s
    for seq, slot in orc.seq_slot.items():
        rc, ls, init = L.lsc_pc_sequence(pc, seq)
        assert rc == L.LSC_OK and (ls, init) == (slot, int(orc.seq_initialized[seq])), seq
    assert L.lsc_pc_counts(pc) == (L.LSC_OK, orc.counts())


def both(lib_call, orc_call):
    """Run one operation on both sides; the outcomes must agree."""
    try:
        expect = orc_call()
        err = None
    except PrefixCacheError as e:
        expect, err = None, e
    got = lib_call()
    rc = got[0] if isinstance(got, tuple) else got
    if err is not None:
        assert rc == KIND_CODE[err.kind], (rc, err)
        return None
    assert rc == L.LSC_OK, L.lsc_error_string(rc)
    return got, expect


def test_worked_example_through_the_abi(lib_cache):
    """§3.1-§3.2 slot 7 -> replacement 9 (tests/golden/promotion_handoff.txt)."""
    g = golden_kv("promotion_handoff.txt")
    pc = lib_cache(g["num_slots"], 16)
    for i in range(g["num_slots"] - 1):
        assert L.lsc_pc_allocate_live_slot(pc, 100 + i) == (L.LSC_OK, i)
    seq = 100 + g["live_slot_before"]
    rc, ops, init, rep = L.lsc_pc_resolve(pc, L.pc_rows([seq], [0], [0xABC], [32]))
    assert rc == L.LSC_OK and rep.save == 1
    assert ops[0]["linear_state_id"] == g["op_linear_state_id"]
    assert ops[0]["save_dst_slot_id"] == g["op_save_dst_slot_id"]
    assert L.lsc_pc_slot(pc, g["replacement_slot"])[1] == L.LSC_SLOT_RESERVED
    assert L.lsc_pc_commit(pc) == L.LSC_OK
    assert L.lsc_pc_sequence(pc, seq) == (L.LSC_OK, g["sequence_slot_after"], g["sequence_initialized_after"])
    assert L.lsc_pc_slot(pc, g["checkpoint_slot_after"])[1:] == (L.LSC_SLOT_CHECKPOINT, 0, 0xABC)
    assert L.lsc_pc_match(pc, 0xABC) == (L.LSC_OK, g["match_after"])


def test_argument_errors(lib_cache):
    pc = lib_cache(4, 16)
    assert L.lsc_pc_create(0, 16)[0] == L.LSC_ERR_INVALID_ARG
    assert L.lsc_pc_create(4, 0)[0] == L.LSC_ERR_INVALID_ARG
    assert L.lsc_pc_unpin(pc, 7) == L.LSC_ERR_OUT_OF_RANGE
    assert L.lsc_pc_unpin(pc, 0) == L.LSC_ERR_INVALID_ARG
    assert L.lsc_pc_slot(pc, -1)[0] == L.LSC_ERR_OUT_OF_RANGE
    assert L.lsc_pc_sequence(pc, 5)[0] == L.LSC_ERR_INVALID_ARG
    assert L.lsc_pc_release_sequence(pc, 5) == L.LSC_ERR_INVALID_ARG
    assert L.lsc_pc_commit(pc) == L.LSC_ERR_ORDER
    assert L.lsc_error_string(L.LSC_ERR_NO_SLOT) != "unknown error"
    # an empty batch is a valid step
    rc, ops, init, rep = L.lsc_pc_resolve(pc, L.pc_rows([], [], [], []))
    assert rc == L.LSC_OK and len(ops) == 0
    assert L.lsc_pc_commit(pc) == L.LSC_OK


def run_random(pc, orc, rng, steps, hashes, max_tokens):
    next_seq = 0
    for _ in range(steps):
        r = rng.random()
        if r < 0.22:
            both(lambda: L.lsc_pc_allocate_live_slot(pc, next_seq), lambda: orc.allocate_live_slot(next_seq))
            next_seq += 1
        elif r < 0.26:   # an already-held sequence: an argument error on both sides
            if orc.seq_slot:
                s = rng.choice(sorted(orc.seq_slot))
                both(lambda: L.lsc_pc_allocate_live_slot(pc, s), lambda: orc.allocate_live_slot(s))
        elif r < 0.34:
            s = rng.choice(sorted(orc.seq_slot) + [10 ** 9]) if orc.seq_slot else 10 ** 9
            both(lambda: L.lsc_pc_release_sequence(pc, s), lambda: orc.release_sequence(s))
        elif r < 0.40:
            h = rng.choice(hashes)
            out = both(lambda: L.lsc_pc_match(pc, h), lambda: orc.match(h))
            assert out[0][1] == out[1]
            if out[1] >= 0 and rng.random() < 0.7:
                both(lambda: L.lsc_pc_unpin(pc, out[1]), lambda: orc.unpin(out[1]))
        elif r < 0.43:
            both(lambda: L.lsc_pc_commit(pc), lambda: orc.commit())
        elif orc.seq_slot:
            seqs = rng.sample(sorted(orc.seq_slot), rng.randint(1, len(orc.seq_slot)))
            if rng.random() < 0.05:
                seqs.append(seqs[0])          # repeated sequence: rejected whole
            rows = [(s, rng.choice(hashes), rng.choice(hashes), rng.randint(0, max_tokens)) for s in seqs]
            arr = L.pc_rows(*zip(*rows))
            out = both(lambda: L.lsc_pc_resolve(pc, arr), lambda: orc.resolve(rows))
            if out is not None:
                (_, ops, init, rep), (eops, einit, erep) = out
                for o, e in zip(ops, eops):
                    assert {k: int(o[k]) for k in L.OP_DTYPE.names} == e
                assert init.tolist() == einit
                assert {k: getattr(rep, k) for k in erep} == erep
                if rng.random() < 0.9:
                    both(lambda: L.lsc_pc_commit(pc), lambda: orc.commit())
        same_state(pc, orc)


@pytest.mark.parametrize("seed", range(8))
def test_random_steps_match_oracle(lib_cache, seed):
    rng = random.Random(seed)
    num_slots = rng.choice([5, 12, 64, 130])
    block = rng.choice([1, 4, 16])
    pc, orc = lib_cache(num_slots, block), PrefixCache(num_slots, block)
    hashes = [0] + [rng.getrandbits(64) | 1 for _ in range(rng.choice([3, 10, 40]))]
    run_random(pc, orc, rng, 400, hashes, 3 * block)


def test_many_slots_and_hashes(lib_cache):
    """A larger id space with structured hash values (the table's probing and
    backward-shift deletion under load)."""
    rng = random.Random(99)
    pc, orc = lib_cache(1000, 8), PrefixCache(1000, 8)
    hashes = [0] + [(i << 32) | 0x1000 for i in range(1, 300)]
    run_random(pc, orc, rng, 600, hashes, 24)
