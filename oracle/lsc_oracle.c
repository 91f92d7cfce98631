/*
 * lsc_oracle.c -- plain CPU oracle for the linear-state prefix cache hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check in
 * __graft_entry__.py and the CPU-baseline leg of bench.py load this library.
 * It shares no source, header, table or constant with the CUDA library; the two
 * sides meet only in the seeded input generators.
 *
 * Everything here is a straight loop in double precision that follows the
 * pages' definitions step by step.  There is no blocking, fusion or reordering
 * beyond what a definition states.  OpenMP only spreads independent rows
 * (or independent (sequence, head) pairs) over the host cores.
 *
 * Sources, cited by page title and section:
 *   [XN] "Linear-State Prefix Cache 内部机制" (xLLM notes)
 *   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复"
 *   [VA] "非连续 KV Cache" (vLLM-Ascend design document)
 *
 * Readings of points the pages leave open are marked READING below.
 *
 * Parity status: every function here is pinned by the not-gpu tests in
 * tests/test_oracle_pins.py (worked example, truth table, invariants, closed
 * forms, brute force in another formulation).  The q/k-head sharing and the
 * L2-norm epsilon are conventions (READING 6, 7) that no page value pins.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- the oracle's own codes (independent of the product library's) ------- */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };
enum { ORC_ATTENTION = 0, ORC_GDN = 1 };
enum {
  ORC_OK = 0,
  ORC_SOFT_COLD = 1,
  ORC_REJECT_ARG = -1,
  ORC_REJECT_RANGE = -2,
  ORC_REJECT_DUP_DST = -3,
  ORC_REJECT_SRC_IS_DST = -4,
  ORC_REJECT_LAYOUT = -5,
};
/* per-row restore decision */
enum { ORC_NOOP = 0, ORC_HIT = 1, ORC_MISS = 2 };

typedef struct {
  int num_layers;
  const int *layer_kind; /* ORC_ATTENTION or ORC_GDN per layer */
  int num_slots;
  int conv_dim, conv_width, conv_dtype;
  int num_v_heads, head_v_dim, head_k_dim, ssm_dtype;
  long long page_bytes;
} orc_pool;

typedef struct {
  long long conv_elems, conv_bytes;   /* one slot's conv state [conv_dim, conv_width-1] */
  long long ssm_elems, ssm_bytes;     /* one slot's ssm state [Hv, dv, dk] */
  long long ssm_offset;               /* byte offset of the ssm view inside a page */
  long long payload;                  /* logical bytes of a page */
  long long page;                     /* physical page stride in bytes */
  long long conv_stride_elems;        /* slot stride of the conv view, in conv elements */
  long long ssm_stride_elems;         /* slot stride of the ssm view, in ssm elements */
  long long region_bytes;             /* one GDN layer: num_slots pages */
  int num_gdn;
} orc_layout_t;

static int elem_size(int dtype) {
  if (dtype == ORC_F32) return 4;
  if (dtype == ORC_BF16 || dtype == ORC_F16) return 2;
  return 0;
}

/*
 * Layout of one GDN layer's region.
 *
 * [VA] §3 ("物理布局与逻辑布局"): a physical page is [logical elements]
 * [alignment padding]; the view's block stride is the physical page size divided
 * by the element size, not the logical size.  [VA] §3.2: the Mamba allocation
 * is exposed as a conv-state view and an SSM-state view, each with its own shape,
 * stride and storage offset, sharing the page stride.  [VA] §3.4 works the
 * numbers: 48 fp16 elements (96 B) in a 128 B page give a stride of 64 elements.
 *
 * READING 1: inside a page the conv state comes first, the ssm state starts at
 * the next 16-byte boundary after it, and the rest of the page is padding.
 * READING 2: the page stride must divide evenly by both element sizes, and must
 * hold the payload.
 */
int orc_layout(const orc_pool *p, orc_layout_t *out) {
  if (!p || !out) return ORC_REJECT_ARG;
  if (p->num_layers <= 0 || p->num_slots <= 0 || !p->layer_kind) return ORC_REJECT_ARG;
  if (p->conv_dim <= 0 || p->conv_width < 2) return ORC_REJECT_ARG;
  if (p->num_v_heads <= 0 || p->head_v_dim <= 0 || p->head_k_dim <= 0) return ORC_REJECT_ARG;
  int esc = elem_size(p->conv_dtype), ess = elem_size(p->ssm_dtype);
  if (!esc || !ess) return ORC_REJECT_ARG;
  int num_gdn = 0;
  for (int l = 0; l < p->num_layers; ++l) {
    if (p->layer_kind[l] == ORC_GDN) num_gdn++;
    else if (p->layer_kind[l] != ORC_ATTENTION) return ORC_REJECT_ARG;
  }
  orc_layout_t L;
  L.conv_elems = (long long)p->conv_dim * (p->conv_width - 1);
  L.conv_bytes = L.conv_elems * esc;
  L.ssm_elems = (long long)p->num_v_heads * p->head_v_dim * p->head_k_dim;
  L.ssm_bytes = L.ssm_elems * ess;
  L.ssm_offset = (L.conv_bytes + 15) / 16 * 16;
  L.payload = L.ssm_offset + L.ssm_bytes;
  L.page = p->page_bytes;
  if (L.page < L.payload) return ORC_REJECT_LAYOUT;
  if (L.page % esc != 0 || L.page % ess != 0) return ORC_REJECT_LAYOUT;
  L.conv_stride_elems = L.page / esc;
  L.ssm_stride_elems = L.page / ess;
  L.region_bytes = (long long)p->num_slots * L.page;
  L.num_gdn = num_gdn;
  *out = L;
  return ORC_OK;
}

/*
 * The has_initial_state gate and the three-way decision, per row.
 *
 * [XN] §5: needs_restore = !linear_state_initialized && n_kv_cache_tokens > 0
 *          && n_kv_cache_tokens % block_size == 0.
 * [XN] §4 (diagram): on a prefix-cache hit the scheduler writes the matched
 *          checkpoint slot into restore_src_slot_id; on a miss it stays -1.
 * [XN] §4.2 (heading only; its body is missing from the page).
 * READING 3: a row that does not need a restore is a no-op; a row that needs
 * one is a hit when restore_src_slot_id >= 0 and a miss otherwise.
 */
static int decide(int initialized, int nkv, int block_size, int src) {
  int needs = !initialized && nkv > 0 && nkv % block_size == 0;
  if (!needs) return ORC_NOOP;
  return src >= 0 ? ORC_HIT : ORC_MISS;
}

/*
 * Validation of the rows that will copy.
 * [XN] §4 (diagram): the worker discovers num_slots and copies by integer slot
 * number; [XN] §1-§2: live slots and checkpoint slots share one id space
 * [0, num_slots), a live slot is private and a checkpoint is frozen.
 * READING 4: for hit rows, both slots must lie in [0, num_slots); two hit rows
 * may not write the same live slot; a source may not be its own destination or
 * another hit row's destination (a frozen checkpoint is never a live slot).
 * Several rows may read one source.  Rows that copy nothing are not checked.
 */
int orc_classify(const orc_pool *p, const int *live_slot, const int *src_slot, int n_rows,
                 const int *nkv, int block_size, const unsigned char *initialized,
                 signed char *action_out) {
  if (!p || n_rows < 0 || block_size <= 0) return ORC_REJECT_ARG;
  if (n_rows > 0 && (!live_slot || !src_slot || !nkv || !initialized)) return ORC_REJECT_ARG;
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  for (int r = 0; r < n_rows; ++r) {
    int a = decide(initialized[r] != 0, nkv[r], block_size, src_slot[r]);
    if (action_out) action_out[r] = (signed char)a;
    if (a != ORC_HIT) continue;
    if (live_slot[r] < 0 || live_slot[r] >= p->num_slots) return ORC_REJECT_RANGE;
    if (src_slot[r] >= p->num_slots) return ORC_REJECT_RANGE;
  }
  for (int r = 0; r < n_rows; ++r) {
    if (decide(initialized[r] != 0, nkv[r], block_size, src_slot[r]) != ORC_HIT) continue;
    if (src_slot[r] == live_slot[r]) return ORC_REJECT_SRC_IS_DST;
    for (int s = 0; s < n_rows; ++s) {
      if (s == r || decide(initialized[s] != 0, nkv[s], block_size, src_slot[s]) != ORC_HIT)
        continue;
      if (s > r && live_slot[s] == live_slot[r]) return ORC_REJECT_DUP_DST;
      if (src_slot[r] == live_slot[s]) return ORC_REJECT_SRC_IS_DST;
    }
  }
  return ORC_OK;
}

/*
 * Worker-side restore.
 *
 * [XN] §4.1: has_initial_state is 1 (warm: use the slot) or 0 (cold: start from
 *          zero); the caller pre-fills it with "this row reused KV tokens"; the
 *          restore only overwrites the entries it must.
 * [XN] §4.3: for every linear layer copy the conv state of the source slot into
 *          the destination slot, and the ssm state likewise; attention layers
 *          own no conv/ssm state and are skipped.  If not a single layer was
 *          copied, the "model has a linear layer" invariant is broken: fall back
 *          to a cold start instead of failing.
 * [KP] "Attention 与 Gated DeltaNet 保存的历史不同": conv and recurrent state of a
 *          restore must come from one history position, so every layer copies
 *          from the same source slot.
 *
 * regions[l] is the host copy of GDN layer l's region (num_slots pages); entries
 * for attention layers are ignored.  On any rejection nothing is modified.
 * READING 5: only the conv view [0, conv_bytes) and the ssm view
 * [ssm_offset, ssm_offset + ssm_bytes) of a page are state; the bytes between
 * them (if any) and the padding up to the page end are never copied.
 */
int orc_restore(const orc_pool *p, unsigned char *const *regions, const int *live_slot,
                const int *src_slot, int n_rows, const int *nkv, int block_size,
                const unsigned char *initialized, unsigned char *has_initial_state) {
  if (n_rows > 0 && !has_initial_state) return ORC_REJECT_ARG;
  int rc = orc_classify(p, live_slot, src_slot, n_rows, nkv, block_size, initialized, NULL);
  if (rc != ORC_OK) return rc;
  orc_layout_t L;
  orc_layout(p, &L);
  for (int l = 0; l < p->num_layers; ++l)
    if (p->layer_kind[l] == ORC_GDN && !regions[l]) return ORC_REJECT_ARG;

  int any_hit = 0;
  for (int r = 0; r < n_rows; ++r) {
    int a = decide(initialized[r] != 0, nkv[r], block_size, src_slot[r]);
    if (a == ORC_MISS) has_initial_state[r] = 0;
    if (a != ORC_HIT) continue;
    any_hit = 1;
    int layers_copied = 0;
    for (int l = 0; l < p->num_layers; ++l) {
      if (p->layer_kind[l] != ORC_GDN) continue; /* attention: nothing to copy */
      unsigned char *dst = regions[l] + (long long)live_slot[r] * L.page;
      const unsigned char *src = regions[l] + (long long)src_slot[r] * L.page;
      memcpy(dst, src, (size_t)L.conv_bytes);
      memcpy(dst + L.ssm_offset, src + L.ssm_offset, (size_t)L.ssm_bytes);
      layers_copied++;
    }
    has_initial_state[r] = layers_copied > 0 ? 1 : 0;
  }
  return (any_hit && L.num_gdn == 0) ? ORC_SOFT_COLD : ORC_OK;
}

/* ---- element access ----------------------------------------------------- */

static double load_elem(const unsigned char *base, int dtype, long long i) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, base + 4 * i, 4);
    return (double)f;
  }
  /* bf16: the upper 16 bits of an IEEE binary32 */
  uint16_t h;
  memcpy(&h, base + 2 * i, 2);
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/*
 * Store a double at the state's precision.
 * READING 8: binary32 storage takes the nearest float; bf16 storage rounds the
 * binary32 value to nearest, ties to even, on its bit pattern (NaN stays NaN).
 */
static void store_elem(unsigned char *base, int dtype, long long i, double v) {
  float f = (float)v;
  if (dtype == ORC_F32) {
    memcpy(base + 4 * i, &f, 4);
    return;
  }
  uint32_t bits;
  memcpy(&bits, &f, 4);
  uint16_t h;
  if ((bits & 0x7f800000u) == 0x7f800000u && (bits & 0x007fffffu)) {
    h = (uint16_t)((bits >> 16) | 0x0040u);
  } else {
    uint32_t lsb = (bits >> 16) & 1u;
    h = (uint16_t)((bits + 0x7fffu + lsb) >> 16);
  }
  memcpy(base + 2 * i, &h, 2);
}

/* exported for the pins: round a binary32 to bf16 bits as store_elem does */
unsigned short orc_bf16_bits(float f) {
  unsigned char b[2];
  store_elem(b, ORC_BF16, 0, (double)f);
  uint16_t h;
  memcpy(&h, b, 2);
  return h;
}

/*
 * Gather: indexed strided rows -> dense tensors.
 * [VA] §4 (gather_ssm_states) and §5: requested state rows are collected into a
 * kernel-friendly tensor; the index mapping and the has_initial_state mask are
 * kept and the padding between pages is not.
 * READING 9: a row whose index is negative, or whose has_initial_state is 0,
 * gathers zeros (cold).  has_init may be NULL (every row warm).
 * conv_dense is [n, conv_dim, conv_width-1], ssm_dense [n, Hv, dv, dk], both
 * at the pool's dtypes.
 */
int orc_gather(const orc_pool *p, const unsigned char *region, const int *idx,
               const unsigned char *has_init, int n, unsigned char *conv_dense,
               unsigned char *ssm_dense) {
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  if (n < 0 || (n > 0 && (!region || !idx || !conv_dense || !ssm_dense))) return ORC_REJECT_ARG;
  for (int i = 0; i < n; ++i)
    if (idx[i] >= p->num_slots) return ORC_REJECT_RANGE;
  for (int i = 0; i < n; ++i) {
    unsigned char *cd = conv_dense + (long long)i * L.conv_bytes;
    unsigned char *sd = ssm_dense + (long long)i * L.ssm_bytes;
    int warm = idx[i] >= 0 && (!has_init || has_init[i] != 0);
    if (warm) {
      const unsigned char *page = region + (long long)idx[i] * L.page;
      memcpy(cd, page, (size_t)L.conv_bytes);
      memcpy(sd, page + L.ssm_offset, (size_t)L.ssm_bytes);
    } else {
      memset(cd, 0, (size_t)L.conv_bytes);
      memset(sd, 0, (size_t)L.ssm_bytes);
    }
  }
  return ORC_OK;
}

/*
 * Scatter: dense tensors -> the strided rows they came from, in place.
 * [VA] §4 (scatter_ssm_states_) and §5: updated rows are written back into the
 * original allocation; padding between pages stays as it was.
 * READING 9: rows with a negative index are skipped; two rows may not name the
 * same slot (the result would depend on order).
 */
int orc_scatter(const orc_pool *p, unsigned char *region, const int *idx, int n,
                const unsigned char *conv_dense, const unsigned char *ssm_dense) {
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  if (n < 0 || (n > 0 && (!region || !idx || !conv_dense || !ssm_dense))) return ORC_REJECT_ARG;
  for (int i = 0; i < n; ++i) {
    if (idx[i] >= p->num_slots) return ORC_REJECT_RANGE;
    for (int j = 0; j < i; ++j)
      if (idx[i] >= 0 && idx[j] == idx[i]) return ORC_REJECT_DUP_DST;
  }
  for (int i = 0; i < n; ++i) {
    if (idx[i] < 0) continue;
    unsigned char *page = region + (long long)idx[i] * L.page;
    memcpy(page, conv_dense + (long long)i * L.conv_bytes, (size_t)L.conv_bytes);
    memcpy(page + L.ssm_offset, ssm_dense + (long long)i * L.ssm_bytes, (size_t)L.ssm_bytes);
  }
  return ORC_OK;
}

/* SiLU(z) = z * sigmoid(z) */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One gated-delta-rule token on one head, in place on S [dv x dk] (double).
 *
 * [KP] "Attention 与 Gated DeltaNet 保存的历史不同": the gate decides how much
 * of the old state is kept; the state's prediction for the current k is compared
 * with the current v and the difference corrects the state; q then reads the
 * updated state.  In symbols (the rule the benchmark spec fixes):
 *   S' = alpha * S (I - beta k k^T) + beta v k^T,   o = S' q.
 * Taken in the order of the description: gate, predict, correct, query.
 */
static void delta_rule_token(double *S, int dv, int dk, const double *q, const double *k,
                             const double *v, double alpha, double beta, double *o) {
  for (int i = 0; i < dv * dk; ++i) S[i] *= alpha;           /* gate */
  for (int r = 0; r < dv; ++r) {
    double pred = 0.0;                                        /* (alpha S) k */
    for (int c = 0; c < dk; ++c) pred += S[r * dk + c] * k[c];
    double err = v[r] - pred;                                 /* compare with v */
    for (int c = 0; c < dk; ++c) S[r * dk + c] += beta * err * k[c]; /* correct */
  }
  for (int r = 0; r < dv; ++r) {                             /* query */
    double acc = 0.0;
    for (int c = 0; c < dk; ++c) acc += S[r * dk + c] * q[c];
    o[r] = acc;
  }
}

/* x / sqrt(sum x^2 + eps), READING 7: eps = 1e-6 inside the square root */
static void l2_normalise(double *x, int n) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss + 1e-6);
  for (int i = 0; i < n; ++i) x[i] *= inv;
}

/*
 * One decode token for n rows of one GDN layer: strided gather -> causal
 * conv1d update -> gated delta rule -> in-place scatter.
 *
 * [VA] §5: state indices -> strided physical state -> gather -> the FLA kernel
 *   -> scatter back into the strided physical state.
 * [VA] §6: the decode step uses causal_conv1d_update and
 *   recurrent_gated_delta_rule.
 *
 * causal_conv1d_update, READING 10: the conv state of channel c holds the last
 * W-1 inputs, oldest first.  The window is [state_c, x_c]; the output is
 * SiLU(sum_j w[c][j] * window[j]) with no bias; the new state is the window's
 * last W-1 entries (the old state shifted by one, x_c appended).
 * READING 6: channels are [q | k | v], each head-major (q, k: Hk heads of dk;
 * v: Hv heads of dv); v head h reads q/k head h / (Hv / Hk).
 * READING 7: q and k of each head are L2-normalised after the conv.
 * READING 9: has_init[i] == 0 reads both states as zero; idx[i] < 0 writes a zero
 * output and touches no state.  Rows must name distinct slots.
 *
 * x [n, conv_dim] and conv_w [conv_dim, conv_width] at the conv dtype; alpha,
 * beta [n, Hv] binary32; out [n, Hv, dv] binary32.
 */
int orc_gdn_decode(const orc_pool *p, unsigned char *region, int n, const int *idx,
                   const unsigned char *has_init, const unsigned char *x,
                   const unsigned char *conv_w, int num_k_heads, const float *alpha,
                   const float *beta, float *out) {
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  const int C = p->conv_dim, W = p->conv_width, Hv = p->num_v_heads;
  const int dv = p->head_v_dim, dk = p->head_k_dim, Hk = num_k_heads;
  if (p->conv_dtype == ORC_F16 || p->ssm_dtype == ORC_F16) return ORC_REJECT_ARG;
  if (Hk <= 0 || Hv % Hk != 0 || C != 2 * Hk * dk + Hv * dv) return ORC_REJECT_ARG;
  if (n < 0 || (n > 0 && (!region || !idx || !x || !conv_w || !alpha || !beta || !out)))
    return ORC_REJECT_ARG;
  for (int i = 0; i < n; ++i) {
    if (idx[i] >= p->num_slots) return ORC_REJECT_RANGE;
    for (int j = 0; j < i; ++j)
      if (idx[i] >= 0 && idx[j] == idx[i]) return ORC_REJECT_DUP_DST;
  }
  const int group = Hv / Hk;

#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n; ++i) {
    float *o_row = out + (long long)i * Hv * dv;
    if (idx[i] < 0) {
      for (int e = 0; e < Hv * dv; ++e) o_row[e] = 0.0f;
      continue;
    }
    int warm = !has_init || has_init[i] != 0;
    unsigned char *page = region + (long long)idx[i] * L.page;
    unsigned char *conv_state = page;
    unsigned char *ssm_state = page + L.ssm_offset;
    const unsigned char *x_row = x + (long long)i * C * elem_size(p->conv_dtype);

    double *y = (double *)malloc(sizeof(double) * C);
    double *window = (double *)malloc(sizeof(double) * W);
    for (int c = 0; c < C; ++c) {
      for (int j = 0; j < W - 1; ++j)
        window[j] = warm ? load_elem(conv_state, p->conv_dtype, (long long)c * (W - 1) + j) : 0.0;
      window[W - 1] = load_elem(x_row, p->conv_dtype, c);
      double z = 0.0;
      for (int j = 0; j < W; ++j) z += load_elem(conv_w, p->conv_dtype, (long long)c * W + j) * window[j];
      y[c] = silu(z);
      for (int j = 0; j < W - 1; ++j)
        store_elem(conv_state, p->conv_dtype, (long long)c * (W - 1) + j, window[j + 1]);
    }
    double *qn = (double *)malloc(sizeof(double) * Hk * dk);
    double *kn = (double *)malloc(sizeof(double) * Hk * dk);
    for (int e = 0; e < Hk * dk; ++e) {
      qn[e] = y[e];
      kn[e] = y[Hk * dk + e];
    }
    for (int g = 0; g < Hk; ++g) {
      l2_normalise(qn + g * dk, dk);
      l2_normalise(kn + g * dk, dk);
    }
    double *S = (double *)malloc(sizeof(double) * dv * dk);
    double *o = (double *)malloc(sizeof(double) * dv);
    for (int h = 0; h < Hv; ++h) {
      int g = h / group;
      long long base = (long long)h * dv * dk;
      for (int e = 0; e < dv * dk; ++e) S[e] = warm ? load_elem(ssm_state, p->ssm_dtype, base + e) : 0.0;
      const double *vh = y + 2 * Hk * dk + h * dv;
      delta_rule_token(S, dv, dk, qn + g * dk, kn + g * dk, vh, (double)alpha[(long long)i * Hv + h],
                       (double)beta[(long long)i * Hv + h], o);
      for (int e = 0; e < dv * dk; ++e) store_elem(ssm_state, p->ssm_dtype, base + e, S[e]);
      for (int r = 0; r < dv; ++r) o_row[h * dv + r] = (float)o[r];
    }
    free(o);
    free(S);
    free(kn);
    free(qn);
    free(window);
    free(y);
  }
  return ORC_OK;
}

/*
 * Token-by-token recurrence of a resumed prefill, for one GDN layer.
 *
 * [KP] "相同前缀不一定能全部复用" and "混合架构需要同时保存 KV 缓存和递归状态":
 * the engine restores the deepest checkpoint and continues the prefill from
 * there, so the recurrence starts from the restored state.
 * [VA] §6: recurrent_gated_delta_rule.
 * READING 11: inputs are post-conv (no conv stage); q and k are used as given
 * (the caller normalises them); each sequence i runs tokens
 * cu_seqlens[i] .. cu_seqlens[i+1]-1 in order from the slot's ssm state (zero if
 * has_init[i] == 0) and its final state is written back to the slot; idx[i] < 0
 * gives zero outputs and touches no state.  The conv state is not touched.
 *
 * q, k [T, Hk, dk]; v [T, Hv, dv]; alpha, beta [T, Hv]; out [T, Hv, dv];
 * all binary32.
 */
int orc_gdn_recurrent(const orc_pool *p, unsigned char *region, int n_seq, const int *idx,
                      const unsigned char *has_init, const int *cu_seqlens, int num_k_heads,
                      const float *q, const float *k, const float *v, const float *alpha,
                      const float *beta, float *out) {
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  const int Hv = p->num_v_heads, dv = p->head_v_dim, dk = p->head_k_dim, Hk = num_k_heads;
  if (p->ssm_dtype == ORC_F16) return ORC_REJECT_ARG;
  if (Hk <= 0 || Hv % Hk != 0) return ORC_REJECT_ARG;
  if (n_seq < 0 || (n_seq > 0 && (!region || !idx || !cu_seqlens))) return ORC_REJECT_ARG;
  if (n_seq > 0 && cu_seqlens[0] != 0) return ORC_REJECT_ARG;
  for (int i = 0; i < n_seq; ++i) {
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return ORC_REJECT_ARG;
    if (idx[i] >= p->num_slots) return ORC_REJECT_RANGE;
    for (int j = 0; j < i; ++j)
      if (idx[i] >= 0 && idx[j] == idx[i]) return ORC_REJECT_DUP_DST;
  }
  if (n_seq > 0 && cu_seqlens[n_seq] > 0 && (!q || !k || !v || !alpha || !beta || !out))
    return ORC_REJECT_ARG;
  const int group = Hv / Hk;

#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int i = 0; i < n_seq; ++i) {
    for (int h = 0; h < Hv; ++h) {
      const int t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
      if (idx[i] < 0) {
        for (int t = t0; t < t1; ++t)
          for (int r = 0; r < dv; ++r) out[((long long)t * Hv + h) * dv + r] = 0.0f;
        continue;
      }
      int warm = !has_init || has_init[i] != 0;
      unsigned char *ssm_state = region + (long long)idx[i] * L.page + L.ssm_offset;
      long long base = (long long)h * dv * dk;
      int g = h / group;
      double *S = (double *)malloc(sizeof(double) * dv * dk);
      double *qd = (double *)malloc(sizeof(double) * dk);
      double *kd = (double *)malloc(sizeof(double) * dk);
      double *vd = (double *)malloc(sizeof(double) * dv);
      double *o = (double *)malloc(sizeof(double) * dv);
      for (int e = 0; e < dv * dk; ++e) S[e] = warm ? load_elem(ssm_state, p->ssm_dtype, base + e) : 0.0;
      for (int t = t0; t < t1; ++t) {
        for (int c = 0; c < dk; ++c) {
          qd[c] = q[((long long)t * Hk + g) * dk + c];
          kd[c] = k[((long long)t * Hk + g) * dk + c];
        }
        for (int r = 0; r < dv; ++r) vd[r] = v[((long long)t * Hv + h) * dv + r];
        delta_rule_token(S, dv, dk, qd, kd, vd, alpha[(long long)t * Hv + h], beta[(long long)t * Hv + h], o);
        for (int r = 0; r < dv; ++r) out[((long long)t * Hv + h) * dv + r] = (float)o[r];
      }
      for (int e = 0; e < dv * dk; ++e) store_elem(ssm_state, p->ssm_dtype, base + e, S[e]);
      free(o);
      free(vd);
      free(kd);
      free(qd);
      free(S);
    }
  }
  return ORC_OK;
}

/*
 * Prefill conv of a resumed prefill, for one GDN layer: causal_conv1d over each
 * sequence's tokens from the slot's conv state, then the split into q | k | v
 * and the L2 norm of q and k per head.
 *
 * [VA] §6 names causal_conv1d_fn (the multi-token conv) beside
 * causal_conv1d_update.  [KP] "相同前缀不一定能全部复用": the prefill continues
 * from the restored checkpoint, so the conv starts from the slot's conv state.
 * READING 10 (as in orc_gdn_decode): the conv state of channel c holds the last
 * W-1 inputs, oldest first; token t of a sequence sees the window of its last W
 * inputs [.., x_(t-1), x_t], the inputs before the sequence's first token being
 * the conv state (zero when has_init[i] == 0); y = SiLU(sum_j w[c][j] window[j]),
 * no bias.  After the sequence, the slot's conv state holds the last W-1 entries
 * of [state, x_(t0) .. x_(t1-1)].  READING 6/7: channels [q | k | v] head-major;
 * q and k L2-normalised per head.  idx[i] < 0: zero outputs, no state touched.
 * The ssm state is not touched.
 *
 * x [T, conv_dim] and conv_w [conv_dim, conv_width] at the conv dtype; q, k
 * [T, Hk, dk], v [T, Hv, dv] binary32.
 */
int orc_gdn_prefill_conv(const orc_pool *p, unsigned char *region, int n_seq, const int *idx,
                         const unsigned char *has_init, const int *cu_seqlens, int num_k_heads,
                         const unsigned char *x, const unsigned char *conv_w, float *q, float *k,
                         float *v) {
  orc_layout_t L;
  int rc = orc_layout(p, &L);
  if (rc != ORC_OK) return rc;
  const int C = p->conv_dim, W = p->conv_width, Hv = p->num_v_heads;
  const int dv = p->head_v_dim, dk = p->head_k_dim, Hk = num_k_heads;
  if (p->conv_dtype == ORC_F16) return ORC_REJECT_ARG;
  if (Hk <= 0 || Hv % Hk != 0 || C != 2 * Hk * dk + Hv * dv) return ORC_REJECT_ARG;
  if (n_seq < 0 || (n_seq > 0 && (!region || !idx || !cu_seqlens))) return ORC_REJECT_ARG;
  if (n_seq > 0 && cu_seqlens[0] != 0) return ORC_REJECT_ARG;
  for (int i = 0; i < n_seq; ++i) {
    if (cu_seqlens[i + 1] < cu_seqlens[i]) return ORC_REJECT_ARG;
    if (idx[i] >= p->num_slots) return ORC_REJECT_RANGE;
    for (int j = 0; j < i; ++j)
      if (idx[i] >= 0 && idx[j] == idx[i]) return ORC_REJECT_DUP_DST;
  }
  if (n_seq > 0 && cu_seqlens[n_seq] > 0 && (!x || !conv_w || !q || !k || !v)) return ORC_REJECT_ARG;
  const int es = elem_size(p->conv_dtype);

#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_seq; ++i) {
    const int t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
    if (idx[i] < 0) {
      for (int t = t0; t < t1; ++t) {
        for (int e = 0; e < Hk * dk; ++e) {
          q[(long long)t * Hk * dk + e] = 0.0f;
          k[(long long)t * Hk * dk + e] = 0.0f;
        }
        for (int e = 0; e < Hv * dv; ++e) v[(long long)t * Hv * dv + e] = 0.0f;
      }
      continue;
    }
    int warm = !has_init || has_init[i] != 0;
    unsigned char *conv_state = region + (long long)idx[i] * L.page;
    /* hist[c][j]: the last W-1 inputs of channel c, oldest first */
    double *hist = (double *)malloc(sizeof(double) * C * (W - 1));
    double *y = (double *)malloc(sizeof(double) * C);
    for (int c = 0; c < C; ++c)
      for (int j = 0; j < W - 1; ++j)
        hist[c * (W - 1) + j] = warm ? load_elem(conv_state, p->conv_dtype, (long long)c * (W - 1) + j) : 0.0;
    for (int t = t0; t < t1; ++t) {
      const unsigned char *x_row = x + (long long)t * C * es;
      for (int c = 0; c < C; ++c) {
        const double xt = load_elem(x_row, p->conv_dtype, c);
        double z = 0.0;
        for (int j = 0; j < W - 1; ++j) z += load_elem(conv_w, p->conv_dtype, (long long)c * W + j) * hist[c * (W - 1) + j];
        z += load_elem(conv_w, p->conv_dtype, (long long)c * W + W - 1) * xt;
        y[c] = silu(z);
        for (int j = 0; j + 1 < W - 1; ++j) hist[c * (W - 1) + j] = hist[c * (W - 1) + j + 1];
        hist[c * (W - 1) + W - 2] = xt;
      }
      for (int g = 0; g < Hk; ++g) {
        l2_normalise(y + g * dk, dk);
        l2_normalise(y + Hk * dk + g * dk, dk);
      }
      for (int e = 0; e < Hk * dk; ++e) {
        q[(long long)t * Hk * dk + e] = (float)y[e];
        k[(long long)t * Hk * dk + e] = (float)y[Hk * dk + e];
      }
      for (int e = 0; e < Hv * dv; ++e) v[(long long)t * Hv * dv + e] = (float)y[2 * Hk * dk + e];
    }
    for (int c = 0; c < C; ++c)
      for (int j = 0; j < W - 1; ++j)
        store_elem(conv_state, p->conv_dtype, (long long)c * (W - 1) + j, hist[c * (W - 1) + j]);
    free(y);
    free(hist);
  }
  return ORC_OK;
}

/* ---- attention K/V blocks and copy_prefix -------------------------------- */

/*
 * An attention K/V pool: per attention layer, one allocation of two lanes
 * [K lane][V lane], each lane num_blocks physical pages; a block's logical
 * payload is block_tokens x kv_heads x head_dim elements followed by padding.
 *
 * [VA] §3: the block stride of the view is the physical page size over the
 * element size, not the logical block size; §3.4: the merged two-lane view
 * (2, blocks, block_tokens, kv_heads, head_dim) takes its lane stride and block
 * stride from the physical allocation.
 * READING 12: inside a block, token-major (the §3.4 order); §3 lists
 * [block, kv_head, token, head_dim] for the unmerged view -- the page uses both
 * orders, and the copy of a token prefix below is defined on token rows either
 * way.
 */
typedef struct {
  int num_layers, num_blocks, block_tokens, num_kv_heads, head_dim, dtype;
  long long page_bytes;
} orc_kv_pool;

typedef struct {
  long long row_bytes;          /* one token row: kv_heads x head_dim elements */
  long long payload;            /* block_tokens rows */
  long long page;
  long long block_stride_elems; /* page / element size */
  long long lane_stride_elems;  /* num_blocks pages, in elements */
  long long region_bytes;       /* one layer: 2 lanes */
} orc_kv_layout_t;

int orc_kv_layout(const orc_kv_pool *p, orc_kv_layout_t *out) {
  if (!p || !out || p->num_layers < 0 || p->num_blocks <= 0 || p->block_tokens <= 0 || p->num_kv_heads <= 0 ||
      p->head_dim <= 0)
    return ORC_REJECT_ARG;
  const int es = elem_size(p->dtype);
  if (!es) return ORC_REJECT_ARG;
  orc_kv_layout_t L;
  L.row_bytes = (long long)p->num_kv_heads * p->head_dim * es;
  L.payload = L.row_bytes * p->block_tokens;
  L.page = p->page_bytes;
  if (L.page < L.payload || L.page % es) return ORC_REJECT_LAYOUT;
  L.block_stride_elems = L.page / es;
  L.lane_stride_elems = (long long)p->num_blocks * L.page / es;
  L.region_bytes = 2LL * p->num_blocks * L.page;
  *out = L;
  return ORC_OK;
}

/*
 * copy_prefix: for op r, token rows [0, n_tokens[r]) of block src[r] are copied
 * to block dst[r] in both lanes of every attention layer.
 *
 * [KP] "混合架构需要同时保存 KV 缓存和递归状态" (figure 2): reusing a prefix in
 * another slot copies its KV with copy_prefix, beside the restore of the
 * recurrent state.  READING 13: a prefix of T tokens is given block by block
 * (full blocks, then the partial last one); rows past n_tokens, the block's
 * padding, the source blocks and every other block stay as they were.  Ops with
 * n_tokens == 0 copy nothing and are not checked; copying ops must name blocks
 * in range, distinct destinations, and no source that is a destination.
 */
int orc_copy_prefix(const orc_kv_pool *p, unsigned char *const *regions, const int *src, const int *dst,
                    const int *n_tokens, int n_ops) {
  orc_kv_layout_t L;
  int rc = orc_kv_layout(p, &L);
  if (rc != ORC_OK) return rc;
  if (n_ops < 0 || (n_ops > 0 && (!src || !dst || !n_tokens))) return ORC_REJECT_ARG;
  for (int r = 0; r < n_ops; ++r) {
    if (n_tokens[r] < 0 || n_tokens[r] > p->block_tokens) return ORC_REJECT_ARG;
    if (n_tokens[r] == 0) continue;
    if (src[r] < 0 || src[r] >= p->num_blocks || dst[r] < 0 || dst[r] >= p->num_blocks) return ORC_REJECT_RANGE;
  }
  for (int r = 0; r < n_ops; ++r) {
    if (n_tokens[r] == 0) continue;
    for (int q = 0; q < n_ops; ++q) {
      if (n_tokens[q] == 0) continue;
      if (q < r && dst[q] == dst[r]) return ORC_REJECT_DUP_DST;
      if (src[r] == dst[q]) return ORC_REJECT_SRC_IS_DST;
    }
  }
  for (int l = 0; l < p->num_layers; ++l)
    if (!regions[l]) return ORC_REJECT_ARG;
  for (int r = 0; r < n_ops; ++r)
    for (int l = 0; l < p->num_layers; ++l)
      for (int lane = 0; lane < 2; ++lane) {
        unsigned char *base = regions[l] + (long long)lane * p->num_blocks * L.page;
        for (int t = 0; t < n_tokens[r]; ++t)
          memcpy(base + (long long)dst[r] * L.page + t * L.row_bytes,
                 base + (long long)src[r] * L.page + t * L.row_bytes, (size_t)L.row_bytes);
      }
  return ORC_OK;
}

/* Number of host threads OpenMP will use (reported beside CPU timings). */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
