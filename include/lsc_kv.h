/*
 * lsc_kv.h -- C ABI of liblsc's attention K/V block pool: page-strided K and V
 * views of every attention layer, and copy_prefix, the device copy that moves a
 * reused prefix's K/V rows into another sequence's blocks.
 *
 * Sources, cited by page title and section:
 *   [VA] "非连续 KV Cache" (vLLM-Ascend design document) §3 (block stride =
 *        physical page size / element size; padding skipped by stride), §3.2
 *        (K and V are separate views), §3.4 (the 48-element block example; the
 *        merged two-lane view (2, blocks, block_tokens, kv_heads, head_dim)
 *        whose lane and block strides come from the physical allocation)
 *   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", figure 2 (reusing a prefix
 *        in another slot copies its KV with copy_prefix)
 *
 * Layout: attention layer l owns one region of two lanes, [K lane][V lane];
 * each lane holds num_blocks physical pages; a block's logical payload is
 * block_tokens rows of kv_heads x head_dim elements (token-major, the §3.4
 * order), followed by padding to page_bytes that no call reads or writes.
 * Regions follow one another in layer order.
 *
 * Conventions are those of lsc.h (return codes, host/device pointers, streams,
 * no host sync except create/destroy).
 */
#ifndef LSC_KV_H
#define LSC_KV_H

#include "lsc.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t num_layers;   /* attention layers holding K/V (> 0) */
  int32_t num_blocks;   /* physical blocks per lane (> 0) */
  int32_t block_tokens; /* token rows per block (> 0) */
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t dtype;        /* lsc_dtype */
  int64_t page_bytes;   /* physical page per block: >= payload, multiple of 16 and of the element size */
} lsc_kv_pool_desc;

typedef struct lsc_kv_pool lsc_kv_pool;

/* Typed strided views of one attention layer ([VA] §3.2, §3.4); strides and
 * offsets in elements of dtype. */
typedef struct {
  void *region;            /* device: the layer's [K lane][V lane] */
  int64_t region_bytes;
  void *k;                 /* device: block 0 of the K lane */
  void *v;                 /* device: block 0 of the V lane */
  int64_t shape[4];        /* num_blocks, block_tokens, kv_heads, head_dim */
  int64_t strides[4];      /* page_bytes / es, kv_heads * head_dim, head_dim, 1 */
  int64_t lane_stride;     /* v - k: num_blocks * page_bytes / es (dim 0 of the merged view) */
  int64_t page_bytes, payload_bytes, row_bytes;
  int32_t dtype;
  int32_t reserved;
} lsc_kv_layer_view;

/* One block of a prefix copy: token rows [0, n_tokens) of src_block go to
 * dst_block, in both lanes of every attention layer. */
typedef struct {
  int32_t src_block;
  int32_t dst_block;
  int32_t n_tokens;  /* 0 .. block_tokens; 0 copies nothing */
  int32_t reserved;  /* must be 0 */
} lsc_kv_copy_op;

/* Bytes a pool with this description needs: num_layers * 2 * num_blocks *
 * page_bytes.  Errors: INVALID_ARG, LAYOUT (page smaller than the payload or
 * not a multiple of the element size), MISALIGNED (page not a multiple of 16). */
int lsc_kv_pool_required_bytes(const lsc_kv_pool_desc *desc, size_t *total_bytes);

/* Create a K/V pool; device_base == NULL allocates (cudaMalloc, owned),
 * otherwise the 256-byte-aligned buffer is borrowed.  Without a GPU a borrowed
 * base gives a host-only pool (views work, copies return CUDA).  Errors: as
 * lsc_kv_pool_required_bytes, plus MISALIGNED (base), NO_MEMORY, CUDA. */
int lsc_kv_pool_create(const lsc_kv_pool_desc *desc, void *device_base, size_t base_bytes, lsc_kv_pool **out);
int lsc_kv_pool_destroy(lsc_kv_pool *pool);
/* Errors: OUT_OF_RANGE (layer). */
int lsc_kv_pool_layer_view(const lsc_kv_pool *pool, int32_t layer, lsc_kv_layer_view *out);

/*
 * copy_prefix ([KP] figure 2): for every op with n_tokens > 0, token rows
 * [0, n_tokens) of src_block are copied to dst_block in the K and V lanes of
 * every attention layer; nothing else changes (rows past n_tokens, padding,
 * source blocks, other blocks).  A prefix of T tokens is passed block by block:
 * its full blocks with n_tokens = block_tokens, then the partial last one.
 * One persistent launch per 2560 ops, 16-byte vector copies, on `stream`;
 * `done_event` (may be NULL) is recorded after the last launch.  ops is a host
 * array, read during the call.  bytes_copied (may be NULL) receives the bytes
 * written.  Errors (nothing enqueued): INVALID_ARG (n_tokens outside
 * [0, block_tokens], reserved != 0, NULL ops with n_ops > 0), OUT_OF_RANGE
 * (a block id), DUP_DST (two copying ops share a destination), SRC_IS_DST (a
 * source is a destination of the same call), CUDA.
 */
int lsc_copy_prefix(lsc_kv_pool *pool, const lsc_kv_copy_op *ops, int32_t n_ops, void *stream,
                    void *done_event, int64_t *bytes_copied);

#ifdef __cplusplus
}
#endif

#endif /* LSC_KV_H */
