"""Plain model of the snapshot store of a prefix cache's disk tier.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/ and bench.py's CPU legs
import this module.

Source: "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", sections "SSD 前缀缓存的写入
与读取" and "磁盘缓存的完整性校验与容量管理":
  * files are written to a temporary name with a CRC-32C of the header and of
    the payload, and renamed to the final name once written; a failed write
    removes the temporary file;
  * a read checks the file's identity, the header CRC and the payload CRC; a
    damaged file is dropped together with the entries that depend on it;
  * the capacity is the configured quota; when space is short, make_room first
    removes blocks no entry references, then evicts unpinned entries least
    recently used first; pin / unpin protect entries in use and unpin updates
    their time; dropping an entry decrements its blocks' reference counts and
    blocks still shared by other entries stay; when no room can be made the
    write fails.

CRC-32C (Castagnoli): reflected polynomial 0x82F63B78, initial value and final
xor 0xFFFFFFFF, computed bit by bit here.

Readings where the page is silent (also in the design notes): the file layout
(a 64-byte header: magic "LSCSNAP1", format version, kind, namespace digest,
key, payload bytes (40 bytes), 20 reserved zero bytes, then the CRC-32C of
those 60 bytes; then the payload, then the payload CRC, all little-endian); "blocks" are the stored blobs
(K/V blocks and state snapshots alike) and an entry references blobs; a blob
written with no entry referencing it is unreferenced until an entry takes it;
"recently used" advances on put_entry, pin and unpin; a blob key is written
once (a second put of the same key is refused); reopening a store clears pins
and orders entries by key; make_room runs before a
blob is written and counts file sizes (header + payload + CRC).
"""
import struct

MAGIC = b"LSCSNAP1"
VERSION = 1
HEADER = 64
POLY = 0x82F63B78


def crc32c(data, crc=0):
    crc ^= 0xFFFFFFFF
    for b in bytes(data):
        crc ^= b
        for _ in range(8):
            crc = (crc >> 1) ^ (POLY if crc & 1 else 0)
    return crc ^ 0xFFFFFFFF


def header(kind, namespace, key, nbytes):
    h = MAGIC + struct.pack("<IIQQQ", VERSION, kind, namespace, key, nbytes)   # 8 + 32 = 40 bytes
    h += b"\0" * (HEADER - 4 - len(h))                                         # reserved, zero
    return h + struct.pack("<I", crc32c(h))


def file_bytes(kind, namespace, key, payload):
    return header(kind, namespace, key, len(payload)) + bytes(payload) + struct.pack("<I", crc32c(payload))


def parse(raw, namespace, key):
    """Returns (ok, kind, payload); ok is False for any damage or mismatch."""
    if len(raw) < HEADER + 4 or raw[:8] != MAGIC:
        return False, None, None
    version, kind, ns, k, n = struct.unpack("<IIQQQ", raw[8:40])
    (hcrc,) = struct.unpack("<I", raw[HEADER - 4:HEADER])
    if hcrc != crc32c(raw[:HEADER - 4]) or version != VERSION or ns != namespace or k != key:
        return False, None, None
    if len(raw) != HEADER + n + 4:
        return False, None, None
    payload = raw[HEADER:HEADER + n]
    (pcrc,) = struct.unpack("<I", raw[HEADER + n:])
    if pcrc != crc32c(payload):
        return False, None, None
    return True, kind, payload


class StoreError(Exception):
    def __init__(self, what, kind):
        super().__init__(what)
        self.kind = kind   # "arg", "no_space", "missing", "corrupt"


class Store:
    """The index of a store: blobs (key -> size), entries (key -> blob keys),
    reference counts, pins and last-use times.  File contents live in `files`
    (name -> bytes), a stand-in for the directory."""

    def __init__(self, namespace, quota):
        self.namespace, self.quota = namespace, quota
        self.files = {}
        self.blobs = {}       # key -> file size
        self.refs = {}        # blob key -> number of entries referencing it
        self.entries = {}     # key -> tuple of blob keys
        self.pins = {}        # entry key -> pin count
        self.last = {}        # entry key -> clock
        self.clock = 0

    def used(self):
        return sum(self.blobs.values())

    def _touch(self, e):
        self.clock += 1
        self.last[e] = self.clock

    def _unlink_blob(self, k):
        del self.blobs[k], self.refs[k], self.files[k]

    def _drop_entry(self, e):
        for b in self.entries.pop(e):
            self.refs[b] -= 1
        del self.pins[e], self.last[e]

    def make_room(self, need):
        """Unreferenced blobs first (smallest key first), then unpinned entries
        least recently used first, until need bytes fit under the quota."""
        if self.used() + need <= self.quota:
            return True
        for k in sorted(k for k, r in self.refs.items() if r == 0):
            self._unlink_blob(k)
            if self.used() + need <= self.quota:
                return True
        while self.used() + need > self.quota:
            cand = [e for e in self.entries if self.pins[e] == 0]
            if not cand:
                return False
            e = min(cand, key=lambda x: self.last[x])
            blobs = self.entries[e]
            self._drop_entry(e)
            for b in sorted(set(blobs)):
                if b in self.refs and self.refs[b] == 0:
                    self._unlink_blob(b)
        return True

    def put_blob(self, key, kind, payload):
        if key == 0 or kind == 255 or key in self.blobs:
            raise StoreError("bad blob", "arg")
        size = HEADER + len(payload) + 4
        if not self.make_room(size):
            raise StoreError("no room", "no_space")
        self.files[key] = file_bytes(kind, self.namespace, key, payload)
        self.blobs[key] = size
        self.refs[key] = 0

    def get_blob(self, key):
        if key not in self.blobs:
            raise StoreError("missing", "missing")
        ok, kind, payload = parse(self.files[key], self.namespace, key)
        if not ok:
            self.drop_damaged(key)
            raise StoreError("damaged", "corrupt")
        return kind, payload

    def drop_damaged(self, key):
        for e in [e for e, bl in self.entries.items() if key in bl]:
            self._drop_entry(e)
        self._unlink_blob(key)

    def put_entry(self, key, blob_keys):
        if key == 0 or key in self.entries or any(b not in self.blobs for b in blob_keys):
            raise StoreError("bad entry", "arg")
        self.entries[key] = tuple(blob_keys)
        for b in blob_keys:
            self.refs[b] += 1
        self.pins[key] = 0
        self._touch(key)

    def drop_entry(self, key):
        if key not in self.entries:
            raise StoreError("missing", "missing")
        self._drop_entry(key)

    def pin(self, key):
        if key not in self.entries:
            raise StoreError("missing", "missing")
        self.pins[key] += 1
        self._touch(key)

    def unpin(self, key):
        if key not in self.entries:
            raise StoreError("missing", "missing")
        if self.pins[key] == 0:
            raise StoreError("not pinned", "arg")
        self.pins[key] -= 1
        self._touch(key)

    def reopen(self):
        """The index as a reopened store rebuilds it from the files: pins
        cleared, entries' recency in ascending key order."""
        self.pins = {e: 0 for e in self.entries}
        self.clock = 0
        for e in sorted(self.entries):
            self._touch(e)
