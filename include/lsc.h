/*
 * lsc.h -- C ABI of liblsc, the GB300 (sm_103a) hot path of a linear-state
 * prefix cache for hybrid Attention + Gated DeltaNet (GDN) models.
 *
 * Sources, cited by page title and section:
 *   [XN] "Linear-State Prefix Cache 内部机制" (xLLM notes)
 *   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复"
 *   [VA] "非连续 KV Cache" (vLLM-Ascend design document)
 *
 * Conventions for every call
 * --------------------------
 * - Return value: LSC_OK (0) on success, LSC_SOFT_COLD (+1) for the soft failure
 *   of lsc_restore, a negative LSC_ERR_* otherwise.  When a call returns an
 *   error, it has enqueued nothing and changed no memory.
 * - "host" pointers are read during the call only and may be freed on return.
 *   "device" pointers must stay valid until the work enqueued on the given
 *   stream has completed.
 * - No call synchronises the host with the device, except lsc_pool_create
 *   (when it allocates), lsc_pool_destroy and lsc_pool_status.
 * - Streams and events are cudaStream_t / cudaEvent_t passed as void*; NULL
 *   stream means the legacy default stream.  All device pointers must belong to
 *   the device that was current when the pool was created, and that device must
 *   be current at every call.
 * - Errors found on the device (an index out of range in a device array) never
 *   fault: the offending row is skipped, and the first such error is recorded in
 *   the pool's device status word, read by lsc_pool_status.
 */
#ifndef LSC_H
#define LSC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------- */
#define LSC_OK 0
#define LSC_SOFT_COLD 1             /* restore: no GDN layer, hit rows were set cold */
#define LSC_ERR_INVALID_ARG (-1)    /* null/negative/inconsistent argument */
#define LSC_ERR_OUT_OF_RANGE (-2)   /* slot id outside [0, num_slots), or layer id outside the pool */
#define LSC_ERR_DUP_DST (-3)        /* two restoring rows write one live slot */
#define LSC_ERR_SRC_IS_DST (-4)     /* a source slot is a destination of the same call */
#define LSC_ERR_MISALIGNED (-5)     /* page stride not a multiple of 16 B, base not 256 B aligned, or a
                                       device array not aligned to its element size (q, k of the
                                       recurrence: 16 B) */
#define LSC_ERR_STATELESS_LAYER (-6)/* the layer is an attention layer: it has no state */
#define LSC_ERR_UNSUPPORTED (-7)    /* shape/dtype combination without a kernel */
#define LSC_ERR_CUDA (-8)           /* a CUDA runtime call failed */
#define LSC_ERR_DEV_TIMEOUT (-9)    /* device status: a bounded device wait gave up */
#define LSC_ERR_NO_MEMORY (-10)     /* allocation failed, or the borrowed buffer is too small */
#define LSC_ERR_LAYOUT (-11)        /* page stride smaller than the payload, or not a multiple of an element size */
#define LSC_ERR_WRONG_DEVICE (-12)  /* the current device is not the pool's device */
#define LSC_ERR_NO_SLOT (-13)       /* prefix cache: no free slot and no unpinned checkpoint to reclaim */
#define LSC_ERR_ORDER (-14)         /* prefix cache: call out of step order (resolve/commit/release) */
#define LSC_ERR_NO_SPACE (-15)      /* snapshot store: no room within the quota after make_room */
#define LSC_ERR_CORRUPT (-16)       /* snapshot store: a damaged file (it and its entries were dropped) */
#define LSC_ERR_NOT_FOUND (-17)     /* snapshot store: no such blob or entry */
#define LSC_ERR_IO (-18)            /* snapshot store: a file operation failed */

/* ---- enums -------------------------------------------------------------- */
typedef enum { LSC_LAYER_ATTENTION = 0, LSC_LAYER_GDN = 1 } lsc_layer_kind;
typedef enum { LSC_F32 = 0, LSC_BF16 = 1, LSC_F16 = 2 } lsc_dtype; /* F16: copies only */

/* Content fingerprint of a prefix; opaque to the library, 0 = "not requested".
 * [XN] §6, §6.1. */
typedef uint64_t lsc_prefix_hash;

/*
 * One batch row's scheduler -> worker record.  [XN] §6 defines the fields:
 *   linear_state_id       this row's live slot (overwritten by this step), -1 = none
 *   restore_prefix_hash   prefix to restore from (nonzero = restore requested)
 *   restore_src_slot_id   checkpoint slot that match() resolved, -1 = miss
 *   save_prefix_hash      prefix to checkpoint (nonzero = save requested)
 *   save_dst_slot_id      >= 0 when the resolve stage confirmed a promotion
 * The worker copies restore_src_slot_id -> linear_state_id.  The hashes and the
 * save fields are carried unchanged: saving is a host-side slot hand-off with no
 * device work ([XN] §3, §7.1).  32 bytes, natural alignment.
 */
typedef struct {
  int32_t linear_state_id;
  int32_t restore_src_slot_id;
  lsc_prefix_hash restore_prefix_hash;
  lsc_prefix_hash save_prefix_hash;
  int32_t save_dst_slot_id;
  int32_t reserved; /* must be 0 */
} LinearStateCacheOp;

/*
 * Pool description.  [VA] §3-§4: one physical page per (GDN layer, slot) holds
 * [conv state][ssm state][alignment padding]; views advance by the physical
 * page stride, so padding is skipped by stride and never copied.  Attention
 * layers carry no linear state and own no bytes of the pool.
 *   conv state of a slot: [conv_dim, conv_width - 1] at conv_dtype, row-major,
 *                         oldest input first; at byte 0 of the page
 *   ssm state of a slot:  [num_v_heads, head_v_dim, head_k_dim] at ssm_dtype,
 *                         row-major; at byte round_up(conv bytes, 16) of the page
 *   page_bytes:           physical page stride, >= payload, multiple of 16
 * GDN layer regions (num_slots pages each) follow one another in layer order.
 */
typedef struct {
  int32_t num_layers;
  const int32_t *layer_kinds; /* host [num_layers] of lsc_layer_kind; copied */
  int32_t num_slots;
  int32_t conv_dim;
  int32_t conv_width;
  int32_t conv_dtype; /* lsc_dtype */
  int32_t num_v_heads;
  int32_t head_v_dim;
  int32_t head_k_dim;
  int32_t ssm_dtype;  /* lsc_dtype */
  int64_t page_bytes;
} lsc_pool_desc;

typedef struct lsc_pool lsc_pool;

/* Typed strided views of one GDN layer ([VA] §3.2, §4 _adjust_kv_layout).
 * Shapes and strides are in elements of the view's dtype; storage offsets are
 * in elements from `region`. */
typedef struct {
  void *region;              /* device: first byte of the layer's region */
  int64_t region_bytes;      /* num_slots * page_bytes */
  int32_t gdn_index;         /* position among GDN layers */
  int32_t conv_dtype, ssm_dtype;
  void *conv;                /* device: slot 0's conv state */
  int64_t conv_shape[3];     /* num_slots, conv_dim, conv_width - 1 */
  int64_t conv_strides[3];   /* page_bytes / conv elem, conv_width - 1, 1 */
  int64_t conv_storage_offset;
  void *ssm;                 /* device: slot 0's ssm state */
  int64_t ssm_shape[4];      /* num_slots, Hv, dv, dk */
  int64_t ssm_strides[4];    /* page_bytes / ssm elem, dv*dk, dk, 1 */
  int64_t ssm_storage_offset;
  int64_t page_bytes, payload_bytes, conv_bytes, ssm_offset_bytes, ssm_bytes;
} lsc_layer_view;

/* Host-side counts of one lsc_restore call. */
typedef struct {
  int32_t n_hit, n_miss, n_noop;
  int32_t soft_cold;      /* 1 when hits were set cold because no GDN layer exists */
  int32_t launches;       /* kernel launches enqueued */
  int32_t reserved;
  int64_t bytes_copied;   /* state bytes written (= bytes read) */
} lsc_restore_report;

/* ---- pool ----------------------------------------------------------------- */

/* Bytes a pool with this description needs: (#GDN layers) * num_slots *
 * page_bytes.  Validates the description (same errors as lsc_pool_create).
 * [VA] §3 (block stride = physical page size / element size). */
int lsc_pool_required_bytes(const lsc_pool_desc *desc, size_t *total_bytes);

/* Create a pool.  device_base == NULL: the library allocates the state memory
 * (cudaMalloc) and owns it; contents are undefined.  Otherwise device_base
 * (256 B aligned, base_bytes >= required) is borrowed and must outlive the
 * pool.  The library also allocates a 4-byte device status word and a pinned
 * host word.  With LSC_LOG=1 in the environment, one "[lsc-pool]" line per GDN
 * layer reports page size, state shapes, strides, storage offsets and
 * contiguity ([VA] §7).  Errors: INVALID_ARG, LAYOUT, MISALIGNED, NO_MEMORY, CUDA. */
int lsc_pool_create(const lsc_pool_desc *desc, void *device_base, size_t base_bytes,
                    lsc_pool **out);

/* Free what the pool owns.  Synchronises the device first. */
int lsc_pool_destroy(lsc_pool *pool);

/* Views of a GDN layer.  Errors: OUT_OF_RANGE (layer), STATELESS_LAYER. */
int lsc_pool_layer_view(const lsc_pool *pool, int32_t layer, lsc_layer_view *out);

/* Number of slots of the pool ([XN] §4: the worker discovers num_slots). */
int32_t lsc_pool_num_slots(const lsc_pool *pool);

/* Read and clear the device status word: waits for `stream` (host sync), then
 * stores LSC_OK or the first device-side error code (OUT_OF_RANGE,
 * INVALID_ARG, DEV_TIMEOUT) into *host_status. */
int lsc_pool_status(lsc_pool *pool, void *stream, int32_t *host_status);

/* ---- restore ([XN] §4, §4.1, §4.3, §5) ---------------------------------- */

/*
 * Classify rows without touching the device.  Per row ([XN] §5):
 *   needs = !linear_state_initialized && n_kv > 0 && n_kv % block_size == 0
 *   !needs                  -> no-op  (action 0)
 *   needs && src >= 0       -> hit    (action 1)
 *   needs && src <  0       -> miss   (action 2)
 * Hit rows are validated: both slots in [0, num_slots) (OUT_OF_RANGE), distinct
 * destinations (DUP_DST), no source equal to any destination (SRC_IS_DST).
 * Several rows may share a source.  Rows that copy nothing are not validated.
 * actions (host [n_rows], may be NULL) and report (may be NULL) are outputs.
 */
int lsc_restore_classify(const lsc_pool *pool, const LinearStateCacheOp *ops, int32_t n_rows,
                         const int32_t *n_kv_cache_tokens, int32_t block_size,
                         const uint8_t *linear_state_initialized, int8_t *actions,
                         lsc_restore_report *report);

/*
 * Worker-side checkpoint restore, enqueued on prepare_stream with no host sync.
 *   ops, n_kv_cache_tokens, linear_state_initialized: host [n_rows]
 *   has_initial_state: device uint8 [n_rows], pre-filled by the caller with
 *       "row reused KV tokens" ([XN] §4.1).  The restore writes hit -> 1,
 *       miss -> 0 and leaves no-op rows unchanged.
 * For every hit row and every GDN layer, the conv view and the ssm view of page
 * restore_src_slot_id are copied to page linear_state_id -- bit-exact, padding
 * and every other byte untouched ([XN] §4.3; one source position for all
 * layers, [KP]).  All layers and rows go in one persistent kernel launch (more
 * launches only when a call has over 2048 hit rows or 3584 has_initial_state
 * writes).  Soft failure ([XN] §4.3): when the pool has no GDN layer, hit rows
 * are set cold (0) and LSC_SOFT_COLD is returned; nothing is copied.
 * If done_event is not NULL it is recorded on prepare_stream after the work,
 * for the forward stream to wait on ([XN] §4.3).
 * Errors: as lsc_restore_classify, plus CUDA; nothing is enqueued on error.
 */
int lsc_restore(lsc_pool *pool, const LinearStateCacheOp *ops, int32_t n_rows,
                const int32_t *n_kv_cache_tokens, int32_t block_size,
                const uint8_t *linear_state_initialized, uint8_t *has_initial_state,
                void *prepare_stream, void *done_event, lsc_restore_report *report);

/* ---- state access ([VA] §4 gather_ssm_states / scatter_ssm_states_, §5) ---- */

/*
 * Strided slots -> dense tensors, for layer `layer` (a GDN layer).
 *   idx: device int32 [n]; has_init: device uint8 [n] or NULL (all warm)
 *   conv_dense: device [n, conv_dim, conv_width-1] at conv_dtype
 *   ssm_dense:  device [n, Hv, dv, dk] at ssm_dtype
 * Row i receives slot idx[i] when idx[i] >= 0 and has_init[i] != 0, zeros
 * otherwise.  idx[i] >= num_slots: zeros, and OUT_OF_RANGE in the status word.
 */
int lsc_gather(lsc_pool *pool, int32_t layer, const int32_t *idx, const uint8_t *has_init,
               int32_t n, void *conv_dense, void *ssm_dense, void *stream);

/*
 * Dense tensors -> strided slots, in place.  Rows with idx[i] < 0 are skipped;
 * only the conv and ssm views of the named pages are written.  Entries of idx
 * that are >= 0 must be distinct (duplicates race).  idx[i] >= num_slots: row
 * skipped, OUT_OF_RANGE in the status word.
 */
int lsc_scatter(lsc_pool *pool, int32_t layer, const int32_t *idx, int32_t n,
                const void *conv_dense, const void *ssm_dense, void *stream);

/* ---- GDN decode step ([VA] §5 access flow, §6 FLA ops; [KP] delta rule) ---- */

typedef struct {
  int32_t n;                /* rows */
  int32_t num_k_heads;      /* Hk; Hv % Hk == 0, conv_dim == 2*Hk*dk + Hv*dv */
  const int32_t *idx;       /* device [n]: live slot of each row, < 0 = padding row */
  const uint8_t *has_init;  /* device [n] or NULL (all warm) */
  const void *x;            /* device [n, conv_dim] at conv_dtype: this token's input */
  const void *conv_weight;  /* device [conv_dim, conv_width] at conv_dtype */
  const float *alpha;       /* device [n, Hv]: gate, already activated */
  const float *beta;        /* device [n, Hv]: write strength, already activated */
  float *out;               /* device [n, Hv, dv] */
  uint32_t flags;           /* 0 or LSC_DECODE_EARLY_STATE; other bits: INVALID_ARG */
} lsc_gdn_decode_args;

/* Flag of lsc_gdn_decode_args.  The decode kernel is launched with programmatic
 * stream serialisation: its CTAs may start on SMs that the previous kernel of
 * the stream has left, and wait for that kernel to complete before reading any
 * input.  With this flag they read idx, has_init and the first state tiles of
 * the layer's rows before that wait, so the state stream of this layer overlaps
 * the end of the previous kernel.  Set it only when the kernel enqueued just
 * before the call on the stream (with no event wait or copy between them)
 * writes none of idx, has_init and the layer's ssm state of those rows -- for
 * example the decode of another layer.  All other inputs are read after the
 * wait, as without the flag. */
#define LSC_DECODE_EARLY_STATE 1u

/*
 * One decode token for n rows of GDN layer `layer`, in one fused kernel that
 * reads and writes the slots through the page stride (gather -> conv update ->
 * gated delta rule -> scatter, [VA] §5):
 *   window_c = [conv_state_c, x_c] (oldest first), y_c = SiLU(sum_j w_cj window_cj),
 *   conv_state_c <- window_c[1:]  (causal_conv1d_update, no bias)
 *   q, k, v = y split [Hk*dk | Hk*dk | Hv*dv], head-major; q, k of each head
 *   L2-normalised with eps 1e-6 inside the square root; v head h uses q/k head
 *   h / (Hv/Hk)
 *   S <- alpha S (I - beta k k^T) + beta v k^T,  out = S q   (per v head)
 * Arithmetic in fp32; states stored back at their dtype (bf16: round to
 * nearest even).  has_init[i] == 0 reads both states as zero.  idx[i] < 0
 * writes zeros to out[i] and touches no state.  If a bounded device wait
 * expires (LSC_ERR_DEV_TIMEOUT in the status word), the states and outputs of
 * the call's rows are unspecified; nothing outside their views is written.  Entries of idx that are >= 0
 * must be distinct.  Supported: head_k_dim in {16, 32, 64, 128}, head_v_dim <=
 * 128, Hv/Hk <= 8, conv_width <= 8, ssm dtype f32 or bf16, conv dtype f32 or
 * bf16; else UNSUPPORTED.  Every device array must be aligned to its element
 * size (MISALIGNED).
 */
int lsc_gdn_decode(lsc_pool *pool, int32_t layer, const lsc_gdn_decode_args *args, void *stream);

typedef struct {
  int32_t n_seq;
  int32_t num_k_heads;
  int32_t total_tokens;      /* == cu_seqlens[n_seq] (host copy, sizes the launch) */
  int32_t algorithm;         /* LSC_RECURRENT_AUTO (0), _TOKEN or _CHUNKED */
  const int32_t *idx;        /* device [n_seq]: live slot, < 0 = padding sequence */
  const uint8_t *has_init;   /* device [n_seq] or NULL (all warm) */
  const int32_t *cu_seqlens; /* device [n_seq + 1], cu_seqlens[0] == 0, non-decreasing */
  const float *q;            /* device [T, Hk, dk], used as given */
  const float *k;            /* device [T, Hk, dk], used as given */
  const float *v;            /* device [T, Hv, dv] */
  const float *alpha;        /* device [T, Hv] */
  const float *beta;         /* device [T, Hv] */
  float *out;                /* device [T, Hv, dv] */
  void *workspace;           /* chunked order only: device scratch of at least
                                workspace_bytes (lsc_gdn_recurrent_workspace_bytes),
                                16-byte aligned, untouched by others until the call's work
                                on the stream completes; NULL = the library takes it from
                                the device's stream-ordered pool (cudaMallocAsync /
                                cudaFreeAsync on the call's stream) */
  size_t workspace_bytes;
} lsc_gdn_recurrent_args;

/* Evaluation order of lsc_gdn_recurrent (both give the token recurrence's
 * result up to fp32 rounding). */
#define LSC_RECURRENT_AUTO 0    /* the library's choice: CHUNKED for head_k_dim 128 (the faster
                                   one there), TOKEN otherwise */
#define LSC_RECURRENT_TOKEN 1   /* one token at a time */
#define LSC_RECURRENT_CHUNKED 2 /* 64 tokens at a time on the tensor cores: the token recurrence
                                   rearranged into per-chunk products (head_k_dim 128 only);
                                   needs a workspace (see lsc_gdn_recurrent_workspace_bytes) */

/*
 * Gated delta rule of a resumed prefill ([KP] "相同前缀不一定能全部复用":
 * continue from the restored checkpoint), for GDN layer `layer`: sequence i
 * runs its tokens in order from slot idx[i]'s ssm state (zero when
 * has_init[i] == 0), writes out[t] = S_t q_t for each token, and writes its
 * final state back to the slot.  No conv stage; the conv state is untouched.
 * idx[i] < 0: zero outputs, no state touched.  A sequence whose cu_seqlens
 * entries fall outside [0, total_tokens] or decrease is skipped and
 * LSC_ERR_INVALID_ARG is recorded in the status word.  q and k must be 16-byte
 * aligned (MISALIGNED).  algorithm selects the evaluation order (any other
 * value: INVALID_ARG).  Supported: head_k_dim in {16, 32, 64, 128} (CHUNKED:
 * 128 only), head_v_dim <= 128, ssm dtype f32 or bf16; else UNSUPPORTED.
 * The chunked order runs two kernels on the stream: the first writes the
 * state-free records of every chunk into the workspace, the second reads them.
 * A caller workspace that is too small gives INVALID_ARG, one not 16-byte
 * aligned MISALIGNED; a failed stream-ordered allocation NO_MEMORY.  With
 * cu_seqlens not non-decreasing, chunk records of different sequences may
 * share workspace slots, and the results of every sequence of the call are
 * then unspecified (the offending sequence is reported as above).
 */
int lsc_gdn_recurrent(lsc_pool *pool, int32_t layer, const lsc_gdn_recurrent_args *args,
                      void *stream);

/*
 * Device scratch that lsc_gdn_recurrent needs for `args` (its n_seq,
 * total_tokens and algorithm; the pool gives num_v_heads and head_k_dim): 0
 * when the call runs the token order; for the chunked order (CHUNKED, or AUTO
 * with head_k_dim 128) one 33 344-byte record per (64-token chunk slot,
 * v head), with (total_tokens + 63) / 64 + n_seq chunk slots -- the records of
 * the state-free quantities of every chunk (lsc_chunk.h), written by the
 * call's first kernel and read by its second.  Host only, no device work.
 * INVALID_ARG for a NULL pointer or a negative size.
 */
int lsc_gdn_recurrent_workspace_bytes(const lsc_pool *pool, const lsc_gdn_recurrent_args *args,
                                      size_t *bytes);

/*
 * lsc_gdn_recurrent's chunked order without any device allocation, for callers
 * that may not allocate at call time (a serving loop with a fixed device
 * footprint, a host whose own allocator owns the GPU's memory, a path that
 * cannot afford an allocation's synchronisation).  The pages describe no such
 * call; it is a convenience of this library.
 *
 * Same arguments and results as lsc_gdn_recurrent with algorithm CHUNKED
 * (args->algorithm must be AUTO or CHUNKED, args->workspace NULL and
 * args->workspace_bytes 0, else INVALID_ARG; head_k_dim must be 128, else
 * UNSUPPORTED).  The per-chunk records go to a scratch array of 64 MiB that the
 * library keeps in each device's memory for the life of the process; a call
 * whose records need more (lsc_gdn_recurrent_workspace_bytes with CHUNKED)
 * returns NO_MEMORY before any work.  The first call on a device, with that
 * device current, looks up the array's device address (a runtime query, no
 * allocation); make that first call before any stream capture.  All calls
 * share the array: calls whose work may overlap on the GPU race and must be
 * ordered by the caller.
 */
int lsc_gdn_recurrent_noalloc(lsc_pool *pool, int32_t layer, const lsc_gdn_recurrent_args *args,
                              void *stream);

/* Arguments of lsc_gdn_prefill_conv.  T = total_tokens; sequence i owns tokens
 * cu_seqlens[i] .. cu_seqlens[i+1]-1 of x, q, k and v. */
typedef struct {
  int32_t n_seq;
  int32_t num_k_heads;       /* Hk; num_v_heads % Hk == 0, conv_dim == 2 Hk dk + Hv dv */
  int32_t total_tokens;
  int32_t reserved;          /* must be 0 */
  const int32_t *idx;        /* device [n_seq]: slot per sequence, -1 = padding */
  const uint8_t *has_init;   /* device [n_seq]: 1 warm, 0 cold; NULL = all warm */
  const int32_t *cu_seqlens; /* device [n_seq + 1] */
  const void *x;             /* device [T, conv_dim] at the conv dtype */
  const void *conv_weight;   /* device [conv_dim, conv_width] at the conv dtype */
  float *q;                  /* device [T, Hk, dk]: L2-normalised per head */
  float *k;                  /* device [T, Hk, dk]: L2-normalised per head */
  float *v;                  /* device [T, Hv, dv] */
} lsc_gdn_prefill_conv_args;

/*
 * Prefill conv of a resumed prefill for GDN layer `layer` ([VA] §6 names
 * causal_conv1d_fn; [KP] "相同前缀不一定能全部复用": the prefill continues from
 * the restored checkpoint): for each sequence, a depthwise causal conv over its
 * tokens whose first W-1 window inputs come from slot idx[i]'s conv state (zero
 * when has_init[i] == 0); y = SiLU(sum_j w[c][j] window[j]), no bias; y splits
 * into q | k | v (head-major) and q, k are L2-normalised per head (eps 1e-6
 * inside the square root).  The slot's conv state then holds the last W-1
 * entries of [old state, the sequence's x], so a later decode or prefill
 * continues from it; the ssm state is untouched.  idx[i] < 0: zero outputs, no
 * state touched.  Sequences must name distinct slots.  Inconsistent cu_seqlens
 * (outside [0, total_tokens] or decreasing) are skipped and LSC_ERR_INVALID_ARG
 * is recorded in the status word.  Two kernels on `stream`: the conv (outputs)
 * and the conv-state update.  Conv dtype f32 or bf16, conv_width <= 8; the fast
 * path (q/k norm fused) needs conv_dim, head_k_dim and head_v_dim multiples of
 * 8, head_k_dim / 8 a power of two <= 32 and 16-byte aligned x and weights;
 * other shapes run a two-pass path.
 */
int lsc_gdn_prefill_conv(lsc_pool *pool, int32_t layer, const lsc_gdn_prefill_conv_args *args,
                         void *stream);

/* ---- misc ------------------------------------------------------------------- */

/* Static description of an error code. */
const char *lsc_error_string(int code);

/* Build description (target architecture, CUDA version). */
const char *lsc_build_info(void);

#ifdef __cplusplus
}
#endif
#endif /* LSC_H */
