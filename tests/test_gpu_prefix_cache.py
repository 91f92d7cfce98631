"""The prefix cache driving the device path: several scheduler steps in which
lsc_pc_resolve's ops feed lsc_restore, a forward writes every row's live slot
(lsc_scatter of seeded states), and lsc_pc_commit promotes checkpoints that
later sequences restore from.  The library and the oracle run the same steps
side by side -- the cache on the host, the restore and the forward on the GPU
against the CPU oracle -- and every pool byte, has_initial_state entry and op
row must be identical.

Source: xLLM notes "Linear-State Prefix Cache 内部机制" §3-§7.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.prefix_cache import PrefixCache
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool, dev
from _util import oracle_layout, oracle_pool

pytestmark = pytest.mark.gpu


def test_prefix_cache_steps_through_restore_and_forward(lsc):
    w = W.get("c0p")
    w.num_slots = 12
    block = 16
    Lo = oracle_layout(w)
    rng = np.random.default_rng(7)
    rc, pc = L.lsc_pc_create(w.num_slots, block)
    assert rc == L.LSC_OK
    orc = PrefixCache(w.num_slots, block)
    opool = oracle_pool(w)
    with DevPool(w, seed=5, random_padding=True) as P:
        regions = {l: P.host[l].copy() for l in P.gdn_layers}
        tokens = {}        # sequence -> tokens computed
        prefix = {}        # sequence -> prefix family (hash of its first blocks)
        seq_next = 0
        restored_from = []
        for step in range(10):
            # a new sequence joins each step; it shares a prefix family with an
            # earlier one half of the time
            seq = seq_next
            seq_next += 1
            rc, slot = L.lsc_pc_allocate_live_slot(pc, seq)
            if rc == L.LSC_ERR_NO_SLOT:
                break
            assert rc == L.LSC_OK and slot == orc.allocate_live_slot(seq)
            prefix[seq] = int(rng.integers(1, 4))
            tokens[seq] = 0
            # BUILD: every live sequence runs this step
            seqs = sorted(tokens)
            rows, nkv = [], []
            for s in seqs:
                new = tokens[s] == 0
                # a new sequence asks to restore its family's 2-block prefix and
                # reuses those KV tokens; a sequence reaching 2 blocks saves it
                rh = (prefix[s] << 8) | 2 if new else 0
                after = 2 * block if new else tokens[s] + block
                sh = (prefix[s] << 8) | (after // block) if after % block == 0 else 0
                rows.append((s, rh, sh, after))
                nkv.append(2 * block if new else tokens[s])
            arr = L.pc_rows(*zip(*rows))
            rc, ops, init, rep = L.lsc_pc_resolve(pc, arr)
            assert rc == L.LSC_OK
            eops, einit, erep = orc.resolve(rows)
            for o, e in zip(ops, eops):
                assert {k: int(o[k]) for k in L.OP_DTYPE.names} == e
            assert init.tolist() == einit
            # RESTORE on the GPU from the library's ops; the oracle from its own
            hs0 = (np.array(nkv) > 0).astype(np.uint8)
            hs = dev(hs0)
            prep = torch.cuda.Stream()
            prep.wait_stream(torch.cuda.current_stream())
            ev = torch.cuda.Event()
            rc, rrep = L.lsc_restore(P.pool, ops, np.array(nkv, np.int32), block, init, hs, prep, ev)
            assert rc == L.LSC_OK
            torch.cuda.current_stream().wait_event(ev)
            hs_o = hs0.copy()
            live = np.array([e["linear_state_id"] for e in eops], np.int32)
            src = np.array([e["restore_src_slot_id"] for e in eops], np.int32)
            assert oracle.restore(opool, regions, live, src, np.array(nkv, np.int32), block,
                                  np.array(einit, np.uint8), hs_o) == oracle.OK
            np.testing.assert_array_equal(hs.cpu().numpy(), hs_o)
            restored_from += [(int(l), int(s_)) for l, s_, h in zip(live, src, hs_o) if s_ >= 0 and h == 1]
            # FORWARD: every row's live slot gets a new seeded state (scatter)
            for l in P.gdn_layers:
                conv = rng.integers(0, 256, (len(live), Lo["conv_bytes"]), dtype=np.uint8)
                ssm = rng.integers(0, 256, (len(live), Lo["ssm_bytes"]), dtype=np.uint8)
                assert L.lsc_scatter(P.pool, l, dev(live), len(live), dev(conv), dev(ssm)) == L.LSC_OK
                assert oracle.scatter(opool, regions[l], live, conv, ssm) == oracle.OK
            torch.cuda.synchronize()
            for l in P.gdn_layers:
                np.testing.assert_array_equal(P.download(l), regions[l])
            # COMMIT
            assert L.lsc_pc_commit(pc) == L.LSC_OK
            orc.commit()
            for (s, _, _, after) in rows:
                tokens[s] = after
        assert P.status() == L.LSC_OK
        assert restored_from, "the scenario restored nothing"
        assert orc.counts()[2] > 0, "the scenario promoted nothing"
    assert L.lsc_pc_destroy(pc) == L.LSC_OK
