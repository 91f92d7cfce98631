"""Snapshot store with a device pool: a slot's linear state saved to the store
(device -> host -> checksummed file) and loaded into another slot is bit-exact
in every GDN layer's conv and ssm views, the file's payload is the slot's views
in layer order, padding and other slots are untouched, and a damaged file is
refused without touching the pool.

Source: Kapitsa 源码拆解 05 ("SSD 前缀缓存的写入与读取": the disk copy restores a
slot after it was reused; "磁盘缓存的完整性校验与容量管理").
"""
import os

import numpy as np
import pytest
import torch

from oracle.store import file_bytes
from linear_attention_state_lsc_gb300 import lsc as L
from linear_attention_state_lsc_gb300 import workloads as W

from _gpu import DevPool
from _util import oracle_layout

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["c0p", "s4", "c2"])
def test_save_then_load_into_another_slot(lsc, tmp_path, name):
    w = W.get(name) if name.startswith("c") else W.small(name)
    if name == "c2":
        w.num_slots = 4
    Lo = oracle_layout(w)
    with DevPool(w, seed=9, random_padding=True) as P:
        rc, st = L.lsc_store_open(str(tmp_path), 0xC0FFEE, 1 << 32)
        assert rc == L.LSC_OK
        src, dst = 1, w.num_slots - 1
        assert L.lsc_store_save_state(st, 77, P.pool, src, torch.cuda.current_stream()) == L.LSC_OK
        # the file: header + the slot's views in GDN layer order + CRC
        want = b"".join(bytes(P.host[l].reshape(w.num_slots, -1)[src][:Lo["conv_bytes"]]) +
                        bytes(P.host[l].reshape(w.num_slots, -1)[src][Lo["ssm_offset"]:Lo["ssm_offset"] + Lo["ssm_bytes"]])
                        for l in P.gdn_layers)
        path = os.path.join(str(tmp_path), "%016x" % 0xC0FFEE, "b", "%016x" % 77)
        assert open(path, "rb").read() == file_bytes(0, 0xC0FFEE, 77, want)
        assert L.lsc_store_load_state(st, 77, P.pool, dst, torch.cuda.current_stream()) == L.LSC_OK
        for l in P.gdn_layers:
            got = P.download(l).reshape(w.num_slots, -1)
            pre = P.host[l].reshape(w.num_slots, -1)
            exp = pre.copy()
            exp[dst, :Lo["conv_bytes"]] = pre[src, :Lo["conv_bytes"]]
            sl = slice(Lo["ssm_offset"], Lo["ssm_offset"] + Lo["ssm_bytes"])
            exp[dst, sl] = pre[src, sl]
            np.testing.assert_array_equal(got, exp)      # padding and other slots as before
        # a damaged file is refused and nothing in the pool changes
        raw = bytearray(open(path, "rb").read())
        raw[100] ^= 0x40
        open(path, "wb").write(bytes(raw))
        before = [P.download(l).copy() for l in P.gdn_layers]
        assert L.lsc_store_load_state(st, 77, P.pool, 0, torch.cuda.current_stream()) == L.LSC_ERR_CORRUPT
        for l, b in zip(P.gdn_layers, before):
            np.testing.assert_array_equal(P.download(l), b)
        assert L.lsc_store_load_state(st, 77, P.pool, 0, None) == L.LSC_ERR_NOT_FOUND
        assert L.lsc_store_save_state(st, 78, P.pool, w.num_slots, None) == L.LSC_ERR_OUT_OF_RANGE
        L.lsc_store_close(st)


def test_load_refuses_another_layout(lsc, tmp_path):
    a, b = W.get("c0p"), W.small("s4")
    with DevPool(a, seed=1) as Pa, DevPool(b, seed=2) as Pb:
        rc, st = L.lsc_store_open(str(tmp_path), 1, 1 << 30)
        assert L.lsc_store_save_state(st, 5, Pa.pool, 0, None) == L.LSC_OK
        assert L.lsc_store_load_state(st, 5, Pb.pool, 0, None) == L.LSC_ERR_LAYOUT
        L.lsc_store_close(st)
