"""Pins for the snapshot-store oracle (oracle/store.py): CRC-32C against the
published check value and the RFC 3720 (iSCSI) Appendix B.4 test vectors,
damage detection in every part of a file, and the capacity policy of Kapitsa's
disk tier (unreferenced blocks first, then unpinned entries least recently
used, shared blocks kept, pins protect, a write with no room fails) on
hand-built cases.  CPU only.
"""
import pytest

from oracle.store import HEADER, Store, StoreError, crc32c, file_bytes, parse


def test_crc32c_check_value_and_rfc3720_vectors():
    assert crc32c(b"123456789") == 0xE3069283          # the catalogue's check value
    assert crc32c(bytes(32)) == 0x8A9136AA              # RFC 3720 B.4: 32 bytes of zeros
    assert crc32c(b"\xff" * 32) == 0x62A8AB43           # 32 bytes of 0xFF
    assert crc32c(bytes(range(32))) == 0x46DD794E       # 0x00 .. 0x1F
    assert crc32c(bytes(range(31, -1, -1))) == 0x113FDB5C  # 0x1F .. 0x00


def test_crc32c_chains():
    data = bytes(range(200))
    assert crc32c(data[120:], crc32c(data[:120])) == crc32c(data)


def test_file_round_trip_and_every_damage_detected():
    payload = bytes((i * 7) % 251 for i in range(300))
    raw = file_bytes(2, 0xABCDEF, 0x1234, payload)
    assert len(raw) == HEADER + 300 + 4
    assert parse(raw, 0xABCDEF, 0x1234) == (True, 2, payload)
    assert not parse(raw, 0xABCDEE, 0x1234)[0]         # another namespace
    assert not parse(raw, 0xABCDEF, 0x1235)[0]         # another key (file identity)
    assert not parse(raw[:-1], 0xABCDEF, 0x1234)[0]    # truncated
    for pos in (0, 9, 20, 44, HEADER, HEADER + 150, len(raw) - 1):
        bad = bytearray(raw)
        bad[pos] ^= 0x10
        assert not parse(bytes(bad), 0xABCDEF, 0x1234)[0], pos


def test_make_room_unreferenced_blocks_first():
    s = Store(1, quota=3 * (HEADER + 104))
    s.put_blob(10, 0, bytes(100))
    s.put_blob(11, 0, bytes(100))
    s.put_entry(100, [10])
    s.put_blob(12, 0, bytes(100))           # fills the quota
    s.put_blob(13, 0, bytes(100))           # needs room: 11 (unreferenced) goes, not the entry
    assert set(s.blobs) == {10, 12, 13} and 100 in s.entries


def test_make_room_evicts_lru_unpinned_entries_and_keeps_shared_blocks():
    size = HEADER + 104
    s = Store(1, quota=4 * size)
    for k in (1, 2, 3):
        s.put_blob(k, 0, bytes(100))
    s.put_entry(100, [1, 2])                # entries share blob 2
    s.put_entry(101, [2, 3])
    s.pin(100)
    s.unpin(100)                            # 100 now more recent than 101
    s.put_blob(4, 0, bytes(100))            # exactly full
    s.put_entry(102, [4])
    s.put_blob(5, 0, bytes(100))            # evicts 101 (least recent unpinned): 3 goes, 2 stays (shared)
    assert 101 not in s.entries and 100 in s.entries
    assert set(s.blobs) == {1, 2, 4, 5}
    assert s.refs[2] == 1


def test_pinned_entries_are_not_evicted_and_full_store_refuses():
    size = HEADER + 104
    s = Store(1, quota=2 * size)
    s.put_blob(1, 0, bytes(100))
    s.put_blob(2, 0, bytes(100))
    s.put_entry(100, [1])
    s.put_entry(101, [2])
    s.pin(100)
    s.pin(101)
    with pytest.raises(StoreError) as e:
        s.put_blob(3, 0, bytes(100))
    assert e.value.kind == "no_space" and set(s.blobs) == {1, 2}
    s.unpin(101)
    s.put_blob(3, 0, bytes(100))            # 101 evicted now
    assert 101 not in s.entries and set(s.blobs) == {1, 3}


def test_damaged_blob_is_dropped_with_its_entries():
    s = Store(7, quota=1 << 20)
    s.put_blob(1, 0, bytes(100))
    s.put_blob(2, 1, b"x" * 50)
    s.put_entry(100, [1, 2])
    s.put_entry(101, [2])
    s.put_entry(102, [1])
    raw = bytearray(s.files[2])
    raw[HEADER + 10] ^= 1
    s.files[2] = bytes(raw)
    with pytest.raises(StoreError) as e:
        s.get_blob(2)
    assert e.value.kind == "corrupt"
    assert 2 not in s.blobs and set(s.entries) == {102}
    assert s.get_blob(1) == (0, bytes(100))
