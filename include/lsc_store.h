/*
 * lsc_store.h -- C ABI of liblsc's snapshot store: the disk tier of the
 * prefix cache, holding state snapshots and K/V blocks as checksummed files
 * under a byte quota, and the entries that reference them.  Host I/O; two
 * helpers move a pool slot's linear state between the device and the store.
 *
 * Source, cited by page title and section:
 *   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "SSD 前缀缓存的写入与读取"
 *        (entries reference KV blocks and state snapshots; a disk copy stays
 *        usable after the slot is reused) and "磁盘缓存的完整性校验与容量管理"
 *        (temporary file, CRC-32C of header and payload, rename; read checks
 *        identity and both CRCs and drops damaged files with the entries that
 *        depend on them; make_room removes unreferenced blocks first, then
 *        unpinned entries least recently used; pin / unpin; dropping an entry
 *        unreferences its blocks, shared blocks stay; no room = the write fails)
 *        and "读取成本与重新计算成本" (the read path uses up to four threads)
 *
 * File format (little-endian), one file per blob or entry:
 *   bytes 0..7    "LSCSNAP1"
 *   8..11         format version (1)
 *   12..15        kind (0 state snapshot, 1 K/V block, other values free;
 *                 255 = an entry)
 *   16..23        namespace digest (the caller's model / layout fingerprint)
 *   24..31        key
 *   32..39        payload bytes
 *   40..59        reserved, zero
 *   60..63        CRC-32C of bytes 0..59
 *   payload, then the CRC-32C of the payload (4 bytes)
 * An entry's payload is its blob keys (u64 each).  CRC-32C: Castagnoli,
 * reflected polynomial 0x82F63B78, initial value and final xor 0xFFFFFFFF.
 * Files live in <dir>/<namespace>/b (blobs) and <dir>/<namespace>/e
 * (entries), named by key in hex (16 digits each); a write goes to
 * <dir>/<namespace>/tmp first and is renamed into place.  Namespaces (the
 * page's isolation of caches by model, drafter and state layout) never share
 * files.
 *
 * Readings of the page (it leaves these open): keys are caller-chosen nonzero
 * 64-bit values (the page derives them from prefix keys); capacity counts file
 * sizes of blobs; make_room runs before each blob write and removes
 * unreferenced blobs in ascending key order, then evicts unpinned entries
 * least recently used first (recency advances on put_entry, pin, unpin);
 * reopening a store rebuilds its index from the files (headers checked,
 * entries read in full; damaged files removed) and orders entries by key.
 *
 * Return codes of lsc.h; on an error nothing changed unless stated.  A store
 * is not thread-safe.
 *
 * Parallel I/O: a payload of at least two parts is written and read by up to
 * four threads, each on one contiguous part (pwrite / pread at its offset)
 * and checksumming it; the payload CRC is joined from the parts' CRCs
 * (crc(A || B) = crc(A) x^(8|B|) + crc(B) mod the polynomial), so the file
 * format does not change.  The part size is 4 MiB, or LSC_STORE_IO_PART bytes
 * (a positive multiple of 4096) when that is set as the store is opened.
 */
#ifndef LSC_STORE_H
#define LSC_STORE_H

#include "lsc.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lsc_store lsc_store;

typedef struct {
  int64_t used_bytes, quota_bytes;
  int32_t n_blobs, n_entries;
  int32_t n_unreferenced, n_pinned;
} lsc_store_stats;

/* Open (creating directories as needed) a store at dir.  Errors: INVALID_ARG,
 * IO, NO_MEMORY. */
int lsc_store_open(const char *dir, uint64_t namespace_digest, int64_t quota_bytes, lsc_store **out);
int lsc_store_close(lsc_store *store);

/* Write a blob (replacing one with the same key): make_room, then temporary
 * file + rename.  Errors: INVALID_ARG (key 0, kind 255, bytes < 0), NO_SPACE
 * (entries evicted on the way stay evicted), IO. */
int lsc_store_put_blob(lsc_store *store, uint64_t key, int32_t kind, const void *data, int64_t bytes);
/* Read a blob into dst (capacity cap bytes); *bytes = payload size, *kind its
 * kind.  Errors: NOT_FOUND, INVALID_ARG (cap too small: *bytes is still set),
 * CORRUPT (the file and every entry referencing it were dropped), IO. */
int lsc_store_get_blob(lsc_store *store, uint64_t key, void *dst, int64_t cap, int64_t *bytes, int32_t *kind);
/* Payload size of a blob without reading it.  Errors: NOT_FOUND. */
int lsc_store_blob_size(const lsc_store *store, uint64_t key, int64_t *bytes);

/* An entry referencing n blobs (which must exist).  Errors: INVALID_ARG (key 0,
 * key in use, a missing blob), IO. */
int lsc_store_put_entry(lsc_store *store, uint64_t key, const uint64_t *blob_keys, int32_t n);
/* The blob keys of an entry (up to cap; *n = their number).  Errors: NOT_FOUND. */
int lsc_store_get_entry(const lsc_store *store, uint64_t key, uint64_t *blob_keys, int32_t cap, int32_t *n);
/* Remove an entry; its blobs lose one reference (and stay until make_room).
 * Errors: NOT_FOUND, IO. */
int lsc_store_drop_entry(lsc_store *store, uint64_t key);
/* Pins protect an entry from eviction; both update its recency.  Errors:
 * NOT_FOUND; unpin: INVALID_ARG when not pinned. */
int lsc_store_pin(lsc_store *store, uint64_t key);
int lsc_store_unpin(lsc_store *store, uint64_t key);
int lsc_store_stats_get(const lsc_store *store, lsc_store_stats *out);

/* The linear state of pool slot `slot` as a kind-0 blob: the conv and ssm views
 * of every GDN layer in layer order (padding excluded), copied device -> host
 * on `stream` (the call waits for it), then written.  Errors: as put_blob,
 * plus OUT_OF_RANGE (slot), CUDA, NO_MEMORY. */
int lsc_store_save_state(lsc_store *store, uint64_t key, lsc_pool *pool, int32_t slot, void *stream);
/* Read a kind-0 blob and copy it into slot `slot` of the pool (host -> device on
 * `stream`; the call waits).  Errors: as get_blob, plus OUT_OF_RANGE, LAYOUT
 * (the payload size does not match the pool), CUDA, NO_MEMORY. */
int lsc_store_load_state(lsc_store *store, uint64_t key, lsc_pool *pool, int32_t slot, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LSC_STORE_H */
