"""The library's snapshot store (include/lsc_store.h) against the oracle
(oracle/store.py): identical files byte for byte, and the same outcome for every
call of random operation sequences -- puts under a small quota (make_room
evicting), entries, pins, drops, reads of files damaged on disk (dropped with
their entries), and reopening the store from its files.  Host I/O: CPU tests.

Source: Kapitsa 源码拆解 05, "SSD 前缀缓存的写入与读取" and
"磁盘缓存的完整性校验与容量管理".
"""
import os
import random

import pytest

from oracle.store import HEADER, Store, StoreError, file_bytes
from linear_attention_state_lsc_gb300 import lsc as L

KIND_CODE = {"arg": L.LSC_ERR_INVALID_ARG, "no_space": L.LSC_ERR_NO_SPACE, "missing": L.LSC_ERR_NOT_FOUND,
             "corrupt": L.LSC_ERR_CORRUPT}


def ns_dir(d, ns):
    return os.path.join(d, "%016x" % ns)


def blob_path(d, key, ns):
    return os.path.join(ns_dir(d, ns), "b", "%016x" % key)


def both(lib_rc, orc_call):
    try:
        out = orc_call()
        err = None
    except StoreError as e:
        out, err = None, e
    rc = lib_rc() if callable(lib_rc) else lib_rc
    got = rc[0] if isinstance(rc, tuple) else rc
    if err is not None:
        assert got == KIND_CODE[err.kind], (got, err.kind)
    else:
        assert got == L.LSC_OK, L.lsc_error_string(got)
    return rc, out, err


def same_index(s, orc, d):
    d = ns_dir(d, orc.namespace)
    rc, st = L.lsc_store_stats_get(s)
    assert st.used_bytes == orc.used() and st.n_blobs == len(orc.blobs) and st.n_entries == len(orc.entries)
    assert st.n_unreferenced == sum(1 for r in orc.refs.values() if r == 0)
    assert st.n_pinned == sum(1 for p in orc.pins.values() if p > 0)
    assert sorted(int(n, 16) for n in os.listdir(os.path.join(d, "b"))) == sorted(orc.blobs)
    assert sorted(int(n, 16) for n in os.listdir(os.path.join(d, "e"))) == sorted(orc.entries)
    for e, bl in orc.entries.items():
        assert L.lsc_store_get_entry(s, e) == (L.LSC_OK, list(bl))


def test_file_bytes_match_the_oracle_format(lsc, tmp_path):
    d = str(tmp_path)
    rc, s = L.lsc_store_open(d, 0xFEEDBEEF, 1 << 20)
    payload = bytes((i * 13) % 256 for i in range(1000))
    assert L.lsc_store_put_blob(s, 0x1234, 1, payload) == L.LSC_OK
    assert open(blob_path(d, 0x1234, 0xFEEDBEEF), "rb").read() == file_bytes(1, 0xFEEDBEEF, 0x1234, payload)
    assert L.lsc_store_put_blob(s, 0x99, 0, b"") == L.LSC_OK            # empty payload
    assert open(blob_path(d, 0x99, 0xFEEDBEEF), "rb").read() == file_bytes(0, 0xFEEDBEEF, 0x99, b"")
    assert L.lsc_store_put_entry(s, 7, [0x1234, 0x99]) == L.LSC_OK
    ent = open(os.path.join(ns_dir(d, 0xFEEDBEEF), "e", "%016x" % 7), "rb").read()
    want = file_bytes(255, 0xFEEDBEEF, 7, (0x1234).to_bytes(8, "little") + (0x99).to_bytes(8, "little"))
    assert ent == want
    assert os.listdir(os.path.join(ns_dir(d, 0xFEEDBEEF), "tmp")) == []   # renamed into place
    L.lsc_store_close(s)


def test_argument_errors(lsc, tmp_path):
    rc, s = L.lsc_store_open(str(tmp_path), 1, 1 << 20)
    assert L.lsc_store_put_blob(s, 0, 0, b"x") == L.LSC_ERR_INVALID_ARG
    assert L.lsc_store_put_blob(s, 3, 255, b"x") == L.LSC_ERR_INVALID_ARG
    assert L.lsc_store_put_blob(s, 3, 0, b"x") == L.LSC_OK
    assert L.lsc_store_put_blob(s, 3, 0, b"y") == L.LSC_ERR_INVALID_ARG   # written once
    assert L.lsc_store_get_blob(s, 4)[0] == L.LSC_ERR_NOT_FOUND
    assert L.lsc_store_put_entry(s, 9, [3, 4]) == L.LSC_ERR_INVALID_ARG   # missing blob
    assert L.lsc_store_put_entry(s, 9, [3]) == L.LSC_OK
    assert L.lsc_store_put_entry(s, 9, [3]) == L.LSC_ERR_INVALID_ARG      # key in use
    assert L.lsc_store_unpin(s, 9) == L.LSC_ERR_INVALID_ARG
    assert L.lsc_store_pin(s, 8) == L.LSC_ERR_NOT_FOUND
    assert L.lsc_store_drop_entry(s, 8) == L.LSC_ERR_NOT_FOUND
    assert L.lsc_store_open(str(tmp_path / "f" / "g" / "h"), 1, 10)[0] == L.LSC_ERR_IO  # no parent
    L.lsc_store_close(s)


def corrupt(d, key, ns, rng):
    p = blob_path(d, key, ns)
    raw = bytearray(open(p, "rb").read())
    pos = rng.randrange(len(raw))
    raw[pos] ^= 1 << rng.randrange(8)
    open(p, "wb").write(bytes(raw))
    return pos


@pytest.mark.parametrize("seed", range(5))
def test_random_operations_match_oracle(lsc, tmp_path, seed):
    rng = random.Random(seed)
    d = str(tmp_path)
    size = lambda n: HEADER + n + 4
    quota = rng.choice([6, 10, 40]) * size(64)
    ns = rng.getrandbits(64)
    rc, s = L.lsc_store_open(d, ns, quota)
    orc = Store(ns, quota)
    keys = list(range(1, 40))
    ekeys = list(range(100, 120))
    for step in range(250):
        r = rng.random()
        if r < 0.35:
            k = rng.choice(keys)
            payload = bytes(rng.getrandbits(8) for _ in range(rng.choice([0, 10, 64, 130])))
            kind = rng.choice([0, 1])
            both(lambda: L.lsc_store_put_blob(s, k, kind, payload), lambda: orc.put_blob(k, kind, payload))
        elif r < 0.5 and orc.blobs:
            e = rng.choice(ekeys)
            bl = rng.sample(sorted(orc.blobs), rng.randint(1, min(3, len(orc.blobs))))
            if rng.random() < 0.1:
                bl.append(max(keys) + 1)          # a missing blob
            both(lambda: L.lsc_store_put_entry(s, e, bl), lambda: orc.put_entry(e, bl))
        elif r < 0.62:
            e = rng.choice(ekeys)
            both(lambda: L.lsc_store_pin(s, e), lambda: orc.pin(e))
        elif r < 0.72:
            e = rng.choice(ekeys)
            both(lambda: L.lsc_store_unpin(s, e), lambda: orc.unpin(e))
        elif r < 0.78:
            e = rng.choice(ekeys)
            both(lambda: L.lsc_store_drop_entry(s, e), lambda: orc.drop_entry(e))
        elif r < 0.92:
            k = rng.choice(keys)
            if k in orc.blobs and rng.random() < 0.3:   # damage the file on disk (both sides)
                corrupt(d, k, ns, rng)
                orc.files[k] = open(blob_path(d, k, ns), "rb").read()
            rc, out, err = both(lambda: L.lsc_store_get_blob(s, k), lambda: orc.get_blob(k))
            if err is None:
                assert (rc[1], rc[2]) == out
        else:
            L.lsc_store_close(s)
            rc, s = L.lsc_store_open(d, ns, quota)
            assert rc == L.LSC_OK
            orc.reopen()
        same_index(s, orc, d)
    L.lsc_store_close(s)


def test_reopen_drops_files_damaged_on_disk(lsc, tmp_path):
    d = str(tmp_path)
    rc, s = L.lsc_store_open(d, 5, 1 << 20)
    for k in (1, 2, 3):
        assert L.lsc_store_put_blob(s, k, 0, bytes([k]) * 50) == L.LSC_OK
    assert L.lsc_store_put_entry(s, 10, [1, 2]) == L.LSC_OK
    assert L.lsc_store_put_entry(s, 11, [3]) == L.LSC_OK
    L.lsc_store_close(s)
    raw = bytearray(open(blob_path(d, 2, 5), "rb").read())
    raw[20] ^= 0xFF                                    # inside the header: found at open
    open(blob_path(d, 2, 5), "wb").write(bytes(raw))
    rc, s = L.lsc_store_open(d, 5, 1 << 20)
    assert rc == L.LSC_OK
    assert L.lsc_store_get_blob(s, 2)[0] == L.LSC_ERR_NOT_FOUND
    assert L.lsc_store_get_entry(s, 10)[0] == L.LSC_ERR_NOT_FOUND   # it referenced the damaged blob
    assert L.lsc_store_get_entry(s, 11) == (L.LSC_OK, [3])
    assert L.lsc_store_get_blob(s, 1) == (L.LSC_OK, 0, bytes([1]) * 50)
    rc, st = L.lsc_store_stats_get(s)
    assert st.n_blobs == 2 and st.n_unreferenced == 1
    # another namespace sees none of these files and leaves them alone
    L.lsc_store_close(s)
    rc, s = L.lsc_store_open(d, 6, 1 << 20)
    assert L.lsc_store_stats_get(s)[1].n_blobs == 0
    L.lsc_store_close(s)
    rc, s = L.lsc_store_open(d, 5, 1 << 20)
    assert L.lsc_store_stats_get(s)[1].n_blobs == 2
    L.lsc_store_close(s)


@pytest.mark.parametrize("n", [4095, 4096 * 2, 4096 * 3 + 123, 40000, 4096 * 9 + 7])
def test_payload_in_parallel_parts(lsc, tmp_path, monkeypatch, n):
    """[KP] reads the disk tier with up to four threads.  With 4 KiB parts a
    payload is written and read in 1-4 parts by as many threads: the file is
    byte-equal to the oracle's (the CRC joined from the parts' CRCs is the CRC
    of the whole payload), it reads back intact, and a damaged byte in any part
    is found (the blob and its entries are dropped)."""
    monkeypatch.setenv("LSC_STORE_IO_PART", "4096")
    d = str(tmp_path)
    rng = random.Random(n)
    payload = bytes(rng.randrange(256) for _ in range(n))
    for where in [None, 0, n // 3, n // 2, n - 1]:
        rc, s = L.lsc_store_open(d, 0xABC, 1 << 24)
        assert rc == L.LSC_OK
        key = 0x100 + (where if where is not None else 0xFFFF)
        assert L.lsc_store_put_blob(s, key, 2, payload) == L.LSC_OK
        path = blob_path(d, key, 0xABC)
        assert open(path, "rb").read() == file_bytes(2, 0xABC, key, payload)
        if where is None:
            assert L.lsc_store_get_blob(s, key) == (L.LSC_OK, 2, payload)
        else:
            assert L.lsc_store_put_entry(s, 9, [key]) == L.LSC_OK
            with open(path, "r+b") as f:
                f.seek(HEADER + where)
                b = f.read(1)
                f.seek(HEADER + where)
                f.write(bytes([b[0] ^ 0x40]))
            assert L.lsc_store_get_blob(s, key)[0] == L.LSC_ERR_CORRUPT
            assert not os.path.exists(path)
            assert L.lsc_store_get_entry(s, 9)[0] == L.LSC_ERR_NOT_FOUND
        L.lsc_store_close(s)


def test_part_size_setting_is_validated(lsc, tmp_path, monkeypatch):
    """A part size that is not a positive multiple of 4096 falls back to the
    default (payloads below 8 MiB then stay in one part); files are unchanged."""
    for i, bad in enumerate(["0", "-4096", "1000", "junk"]):
        monkeypatch.setenv("LSC_STORE_IO_PART", bad)
        rc, s = L.lsc_store_open(str(tmp_path), 5, 1 << 20)
        assert rc == L.LSC_OK
        payload = bytes(range(256)) * 40
        key = 0x500 + i
        assert L.lsc_store_put_blob(s, key, 1, payload) == L.LSC_OK
        assert open(blob_path(str(tmp_path), key, 5), "rb").read() == file_bytes(1, 5, key, payload)
        assert L.lsc_store_get_blob(s, key) == (L.LSC_OK, 1, payload)
        L.lsc_store_close(s)
