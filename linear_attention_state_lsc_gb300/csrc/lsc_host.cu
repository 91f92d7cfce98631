// lsc_host.cu -- host side of liblsc: pool layout, validation, restore
// classification and plan packing, and the C entry points.
//
// Sources, cited by page title and section:
//   [XN] "Linear-State Prefix Cache 内部机制" (xLLM notes)
//   [VA] "非连续 KV Cache" (vLLM-Ascend design document)
#include <cuda_runtime.h>

#include <algorithm>
#include <initializer_list>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "lsc.h"
#include "lsc_chunk.h"
#include "lsc_internal.h"

#define LSC_STR2(x) #x
#define LSC_STR(x) LSC_STR2(x)

struct lsc_pool {
  int device;
  int num_sms;
  std::vector<int32_t> kinds;
  std::vector<int32_t> gdn_index;  // per layer: position among GDN layers, -1 for attention
  lsc::Geom g;
  size_t base_bytes;
  bool owns_base;
  int32_t *h_status;  // pinned
};

namespace {

int esize(int32_t dtype) {
  switch (dtype) {
    case LSC_F32: return 4;
    case LSC_BF16: return 2;
    case LSC_F16: return 2;
    default: return 0;
  }
}

// Every pointer aligned to `a` bytes (NULL counts as aligned).  Device arrays
// must be aligned to their element size: a misaligned element access faults.
bool all_aligned(std::initializer_list<const void *> ptrs, uintptr_t a) {
  for (const void *q : ptrs)
    if ((uintptr_t)q % a) return false;
  return true;
}

// Bound of every device-side wait (mbarrier), in nanoseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Host-side fault injection for the tests: LSC_FAULT=<name>.
bool fault(const char *name) {
  const char *f = getenv("LSC_FAULT");
  return f && strcmp(f, name) == 0;
}

// [VA] §3: a page is [logical payload][alignment padding]; the block stride is
// the physical page size over the element size.  Inside a page: conv view at 0,
// ssm view at the next 16 B boundary after it.
int describe(const lsc_pool_desc *d, lsc::Geom *g, std::vector<int32_t> *kinds,
             std::vector<int32_t> *gdn_index) {
  if (!d || !d->layer_kinds || d->num_layers <= 0 || d->num_slots <= 0) return LSC_ERR_INVALID_ARG;
  if (d->conv_dim <= 0 || d->conv_width < 2 || d->num_v_heads <= 0 || d->head_v_dim <= 0 ||
      d->head_k_dim <= 0)
    return LSC_ERR_INVALID_ARG;
  const int esc = esize(d->conv_dtype), ess = esize(d->ssm_dtype);
  if (!esc || !ess) return LSC_ERR_INVALID_ARG;
  std::vector<int32_t> k(d->layer_kinds, d->layer_kinds + d->num_layers), gi(d->num_layers, -1);
  int32_t ng = 0;
  for (int l = 0; l < d->num_layers; ++l) {
    if (k[l] == LSC_LAYER_GDN) gi[l] = ng++;
    else if (k[l] != LSC_LAYER_ATTENTION) return LSC_ERR_INVALID_ARG;
  }
  lsc::Geom G{};
  G.conv_bytes = (int64_t)d->conv_dim * (d->conv_width - 1) * esc;
  G.ssm_bytes = (int64_t)d->num_v_heads * d->head_v_dim * d->head_k_dim * ess;
  G.ssm_off = (G.conv_bytes + 15) / 16 * 16;
  G.page = d->page_bytes;
  if (G.page < G.ssm_off + G.ssm_bytes || G.page % esc || G.page % ess) return LSC_ERR_LAYOUT;
  if (G.page % 16) return LSC_ERR_MISALIGNED;
  G.region_bytes = (int64_t)d->num_slots * G.page;
  G.num_slots = d->num_slots;
  G.num_gdn = ng;
  G.conv_dim = d->conv_dim;
  G.conv_width = d->conv_width;
  G.conv_dtype = d->conv_dtype;
  G.Hv = d->num_v_heads;
  G.dv = d->head_v_dim;
  G.dk = d->head_k_dim;
  G.ssm_dtype = d->ssm_dtype;
  if (g) *g = G;
  if (kinds) kinds->swap(k);
  if (gdn_index) gdn_index->swap(gi);
  return LSC_OK;
}

int check_device(const lsc_pool *p) {
  if (p->device < 0) return LSC_ERR_CUDA;  // host-only pool
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LSC_ERR_CUDA;
  return dev == p->device ? LSC_OK : LSC_ERR_WRONG_DEVICE;
}

int layer_base(const lsc_pool *p, int32_t layer, uint8_t **out) {
  if (layer < 0 || layer >= (int32_t)p->kinds.size()) return LSC_ERR_OUT_OF_RANGE;
  if (p->gdn_index[layer] < 0) return LSC_ERR_STATELESS_LAYER;
  *out = p->g.base + (int64_t)p->gdn_index[layer] * p->g.region_bytes;
  return LSC_OK;
}

void log_layout(const lsc_pool *p) {
  const char *e = getenv("LSC_LOG");
  if (!e || strcmp(e, "1") != 0) return;
  const lsc::Geom &g = p->g;
  const int esc = esize(g.conv_dtype), ess = esize(g.ssm_dtype);
  for (size_t l = 0; l < p->kinds.size(); ++l) {
    if (p->gdn_index[l] < 0) continue;
    const int64_t region = (int64_t)p->gdn_index[l] * g.region_bytes;
    const bool contiguous = g.conv_bytes == g.page && g.ssm_bytes == g.page;
    fprintf(stderr,
            "[lsc-pool] layer=%zu gdn=%d page_bytes=%lld conv shape=[%d,%d,%d] stride=[%lld,%d,1] "
            "offset=%lld ssm shape=[%d,%d,%d,%d] stride=[%lld,%d,%d,1] offset=%lld "
            "payload=%lld padding=%lld contiguous=%d\n",
            l, p->gdn_index[l], (long long)g.page, g.num_slots, g.conv_dim, g.conv_width - 1,
            (long long)(g.page / esc), g.conv_width - 1, (long long)(region / esc), g.num_slots, g.Hv,
            g.dv, g.dk, (long long)(g.page / ess), g.dv * g.dk, g.dk,
            (long long)((region + g.ssm_off) / ess), (long long)(g.ssm_off + g.ssm_bytes),
            (long long)(g.page - g.ssm_off - g.ssm_bytes), contiguous ? 1 : 0);
  }
}

// [XN] §5 gate and the per-row decision; [XN] §1-§4 for the validation rules.
int classify(const lsc_pool *p, const LinearStateCacheOp *ops, int32_t n_rows, const int32_t *nkv,
             int32_t block_size, const uint8_t *init, std::vector<int8_t> *actions,
             lsc_restore_report *rep) {
  if (n_rows < 0 || block_size <= 0) return LSC_ERR_INVALID_ARG;
  if (n_rows > 0 && (!ops || !nkv || !init)) return LSC_ERR_INVALID_ARG;
  actions->assign(n_rows, 0);
  const int32_t S = p->g.num_slots;
  lsc_restore_report r{};
  std::vector<uint8_t> is_dst(S, 0);
  for (int32_t i = 0; i < n_rows; ++i) {
    const bool needs = !init[i] && nkv[i] > 0 && nkv[i] % block_size == 0;
    if (!needs) { r.n_noop++; continue; }
    const int32_t src = ops[i].restore_src_slot_id, dst = ops[i].linear_state_id;
    if (src < 0) { (*actions)[i] = 2; r.n_miss++; continue; }
    if (dst < 0 || dst >= S || src >= S) return LSC_ERR_OUT_OF_RANGE;
    if (is_dst[dst]) return LSC_ERR_DUP_DST;
    is_dst[dst] = 1;
    (*actions)[i] = 1;
    r.n_hit++;
  }
  for (int32_t i = 0; i < n_rows; ++i)
    if ((*actions)[i] == 1 && is_dst[ops[i].restore_src_slot_id]) return LSC_ERR_SRC_IS_DST;
  r.soft_cold = (r.n_hit > 0 && p->g.num_gdn == 0) ? 1 : 0;
  if (p->g.num_gdn > 0) r.bytes_copied = (int64_t)r.n_hit * p->g.num_gdn * (p->g.conv_bytes + p->g.ssm_bytes);
  if (rep) *rep = r;
  return LSC_OK;
}

}  // namespace

extern "C" {

const char *lsc_error_string(int code) {
  switch (code) {
    case LSC_OK: return "ok";
    case LSC_SOFT_COLD: return "soft failure: no GDN layer, hit rows set cold";
    case LSC_ERR_INVALID_ARG: return "invalid argument";
    case LSC_ERR_OUT_OF_RANGE: return "slot or layer id out of range";
    case LSC_ERR_DUP_DST: return "two restoring rows share a destination slot";
    case LSC_ERR_SRC_IS_DST: return "a source slot is also a destination";
    case LSC_ERR_MISALIGNED: return "misaligned page stride or base address";
    case LSC_ERR_STATELESS_LAYER: return "attention layer has no linear state";
    case LSC_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case LSC_ERR_CUDA: return "CUDA runtime error";
    case LSC_ERR_DEV_TIMEOUT: return "a bounded device wait gave up";
    case LSC_ERR_NO_MEMORY: return "out of memory or buffer too small";
    case LSC_ERR_LAYOUT: return "page stride smaller than the payload or not a multiple of an element size";
    case LSC_ERR_WRONG_DEVICE: return "current device is not the pool's device";
    case LSC_ERR_NO_SLOT: return "no free slot and no unpinned checkpoint to reclaim";
    case LSC_ERR_ORDER: return "prefix cache call out of step order";
    case LSC_ERR_NO_SPACE: return "snapshot store: no room within the quota";
    case LSC_ERR_CORRUPT: return "snapshot store: damaged file dropped";
    case LSC_ERR_NOT_FOUND: return "snapshot store: no such blob or entry";
    case LSC_ERR_IO: return "snapshot store: file operation failed";
    default: return "unknown error";
  }
}

const char *lsc_build_info(void) {
  return "liblsc sm_103a (CUDA " LSC_STR(__CUDACC_VER_MAJOR__) "." LSC_STR(__CUDACC_VER_MINOR__) ")";
}

int lsc_pool_required_bytes(const lsc_pool_desc *desc, size_t *total_bytes) {
  lsc::Geom g;
  int rc = describe(desc, &g, nullptr, nullptr);
  if (rc != LSC_OK) return rc;
  if (!total_bytes) return LSC_ERR_INVALID_ARG;
  *total_bytes = (size_t)g.num_gdn * (size_t)g.region_bytes;
  return LSC_OK;
}

int lsc_pool_create(const lsc_pool_desc *desc, void *device_base, size_t base_bytes, lsc_pool **out) {
  lsc::TraceRange trace_("lsc_pool_create");
  if (!out) return LSC_ERR_INVALID_ARG;
  *out = nullptr;
  lsc_pool *p = new (std::nothrow) lsc_pool();
  if (!p) return LSC_ERR_NO_MEMORY;
  int rc = describe(desc, &p->g, &p->kinds, &p->gdn_index);
  if (rc != LSC_OK) { delete p; return rc; }
  const size_t need = (size_t)p->g.num_gdn * (size_t)p->g.region_bytes;
  if (device_base) {
    if ((uintptr_t)device_base % 256) { delete p; return LSC_ERR_MISALIGNED; }
    if (base_bytes < need) { delete p; return LSC_ERR_NO_MEMORY; }
  }
  if (fault("alloc")) { delete p; return LSC_ERR_NO_MEMORY; }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    // No GPU: a borrowed base gives a host-only pool (layout, views and
    // classification work; every call that would enqueue returns LSC_ERR_CUDA).
    cudaGetLastError();
    if (!device_base && need > 0) { delete p; return LSC_ERR_CUDA; }
    p->device = -1;
    p->g.base = (uint8_t *)device_base;
    p->base_bytes = base_bytes;
    log_layout(p);
    *out = p;
    return LSC_OK;
  }
  if (cudaGetDevice(&p->device) != cudaSuccess) { delete p; return LSC_ERR_CUDA; }
  if (cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return LSC_ERR_CUDA;
  }
  if (cudaMalloc(&p->g.status, 256) != cudaSuccess) { cudaGetLastError(); delete p; return LSC_ERR_NO_MEMORY; }
  if (cudaMemset(p->g.status, 0, 256) != cudaSuccess ||
      cudaMallocHost(&p->h_status, sizeof(int32_t)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(p->g.status);
    delete p;
    return LSC_ERR_CUDA;
  }
  if (device_base) {
    p->g.base = (uint8_t *)device_base;
    p->base_bytes = base_bytes;
    p->owns_base = false;
  } else if (need > 0) {
    if (cudaMalloc(&p->g.base, need) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(p->g.status);
      cudaFreeHost(p->h_status);
      delete p;
      return LSC_ERR_NO_MEMORY;
    }
    p->base_bytes = need;
    p->owns_base = true;
  }
  log_layout(p);
  *out = p;
  return LSC_OK;
}

int lsc_pool_destroy(lsc_pool *p) {
  if (!p) return LSC_ERR_INVALID_ARG;
  int rc = LSC_OK;
  if (p->device < 0) { delete p; return rc; }
  if (cudaDeviceSynchronize() != cudaSuccess) rc = LSC_ERR_CUDA;
  if (p->owns_base && p->g.base) cudaFree(p->g.base);
  if (p->g.status) cudaFree(p->g.status);
  if (p->h_status) cudaFreeHost(p->h_status);
  delete p;
  return rc;
}

int32_t lsc_pool_num_slots(const lsc_pool *p) { return p ? p->g.num_slots : -1; }

int lsc_pool_layer_view(const lsc_pool *p, int32_t layer, lsc_layer_view *v) {
  if (!p || !v) return LSC_ERR_INVALID_ARG;
  uint8_t *region;
  int rc = layer_base(p, layer, &region);
  if (rc != LSC_OK) return rc;
  const lsc::Geom &g = p->g;
  const int esc = esize(g.conv_dtype), ess = esize(g.ssm_dtype);
  memset(v, 0, sizeof(*v));
  v->region = region;
  v->region_bytes = g.region_bytes;
  v->gdn_index = p->gdn_index[layer];
  v->conv_dtype = g.conv_dtype;
  v->ssm_dtype = g.ssm_dtype;
  v->conv = region;
  v->conv_shape[0] = g.num_slots;
  v->conv_shape[1] = g.conv_dim;
  v->conv_shape[2] = g.conv_width - 1;
  v->conv_strides[0] = g.page / esc;  // [VA] §3: block stride = page size / element size
  v->conv_strides[1] = g.conv_width - 1;
  v->conv_strides[2] = 1;
  v->conv_storage_offset = 0;
  v->ssm = region + g.ssm_off;
  v->ssm_shape[0] = g.num_slots;
  v->ssm_shape[1] = g.Hv;
  v->ssm_shape[2] = g.dv;
  v->ssm_shape[3] = g.dk;
  v->ssm_strides[0] = g.page / ess;
  v->ssm_strides[1] = (int64_t)g.dv * g.dk;
  v->ssm_strides[2] = g.dk;
  v->ssm_strides[3] = 1;
  v->ssm_storage_offset = g.ssm_off / ess;
  v->page_bytes = g.page;
  v->payload_bytes = g.ssm_off + g.ssm_bytes;
  v->conv_bytes = g.conv_bytes;
  v->ssm_offset_bytes = g.ssm_off;
  v->ssm_bytes = g.ssm_bytes;
  return LSC_OK;
}

int lsc_pool_status(lsc_pool *p, void *stream, int32_t *host_status) {
  lsc::TraceRange trace_("lsc_pool_status");
  if (!p || !host_status) return LSC_ERR_INVALID_ARG;
  int rc = check_device(p);
  if (rc != LSC_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(p->h_status, p->g.status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(p->g.status, 0, sizeof(int32_t), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return LSC_ERR_CUDA;
  *host_status = *p->h_status;
  return LSC_OK;
}

int lsc_restore_classify(const lsc_pool *p, const LinearStateCacheOp *ops, int32_t n_rows,
                         const int32_t *nkv, int32_t block_size, const uint8_t *init, int8_t *actions,
                         lsc_restore_report *report) {
  if (!p) return LSC_ERR_INVALID_ARG;
  std::vector<int8_t> act;
  int rc = classify(p, ops, n_rows, nkv, block_size, init, &act, report);
  if (rc != LSC_OK) return rc;
  if (actions && n_rows > 0) memcpy(actions, act.data(), n_rows);
  return LSC_OK;
}

int lsc_restore(lsc_pool *p, const LinearStateCacheOp *ops, int32_t n_rows, const int32_t *nkv,
                int32_t block_size, const uint8_t *init, uint8_t *has_initial_state, void *prepare_stream,
                void *done_event, lsc_restore_report *report) {
  lsc::TraceRange trace_("lsc_restore");
  if (!p) return LSC_ERR_INVALID_ARG;
  std::vector<int8_t> act;
  lsc_restore_report rep{};
  int rc = classify(p, ops, n_rows, nkv, block_size, init, &act, &rep);
  if (rc != LSC_OK) return rc;
  if (rep.n_hit + rep.n_miss > 0 && !has_initial_state) return LSC_ERR_INVALID_ARG;
  rc = check_device(p);
  if (rc != LSC_OK) return rc;
  cudaStream_t stream = (cudaStream_t)prepare_stream;
  const lsc::Geom &g = p->g;

  // Work: hit rows x GDN layers x chunks of the copied byte ranges of a page.
  // When the ssm view starts right after the conv view the two are one range.
  // ~31 KB, passed by value at launch; one per host thread so concurrent callers
  // on different pools do not share it.
  thread_local lsc::RestorePlan plan;
  lsc::RestorePlan &P = plan;
  memset(&P, 0, offsetof(lsc::RestorePlan, hit));
  P.base = g.base;
  P.hs = has_initial_state;
  P.region_bytes = g.region_bytes;
  P.page = g.page;
  P.chunk_bytes = 32 << 10;
  if (g.ssm_off == g.conv_bytes) {
    P.seg_off[0] = 0;
    P.seg_len[0] = g.conv_bytes + g.ssm_bytes;
  } else {
    P.seg_off[0] = 0;
    P.seg_len[0] = g.conv_bytes;
    P.seg_off[1] = g.ssm_off;
    P.seg_len[1] = g.ssm_bytes;
  }
  for (int s = 0; s < 2; ++s) P.seg_chunks[s] = (int32_t)((P.seg_len[s] + P.chunk_bytes - 1) / P.chunk_bytes);
  P.chunks_per_slot = P.seg_chunks[0] + P.seg_chunks[1];
  P.num_gdn = g.num_gdn;
  P.status = g.status;
  // The copy goes through shared memory with 1-D TMA bulk copies when every
  // copied range is 16-byte aligned in offset and length (the bulk copy's
  // rule), else as 16-byte (or narrower) vectors through registers;
  // LSC_RESTORE_COPY=vector selects the vector copy, for measurement.
  const char *mode = getenv("LSC_RESTORE_COPY");
  const bool vector_only = mode && strcmp(mode, "vector") == 0;
  P.bulk = !vector_only && ((P.seg_off[0] | P.seg_len[0] | P.seg_off[1] | P.seg_len[1]) & 15) == 0;

  const int grid = P.bulk ? lsc::restore_bulk_grid(p->num_sms) : lsc::restore_grid(p->num_sms);
  int launches = 0;
  int32_t i = 0;
  while (i < n_rows) {
    P.n_hits = 0;
    P.n_hs = 0;
    for (; i < n_rows; ++i) {
      if (act[i] == 0) continue;
      const bool hit = act[i] == 1;
      if (P.n_hs == lsc::kPlanMaxHs || (hit && g.num_gdn > 0 && P.n_hits == lsc::kPlanMaxHits)) break;
      // [XN] §4.1: hit -> warm (1), miss -> cold (0); [XN] §4.3: with no GDN
      // layer nothing is copied and the hit falls back to cold.
      const int v = (hit && g.num_gdn > 0) ? 1 : 0;
      P.hs_ops[P.n_hs++] = (i << 1) | v;
      if (hit && g.num_gdn > 0) P.hit[P.n_hits++] = make_int2(ops[i].linear_state_id, ops[i].restore_src_slot_id);
    }
    if (P.n_hs == 0) continue;
    {  // does a source slot feed more than one hit of this launch
      std::vector<int32_t> src(P.n_hits);
      for (int32_t h = 0; h < P.n_hits; ++h) src[h] = P.hit[h].y;
      std::sort(src.begin(), src.end());
      P.src_reuse = std::adjacent_find(src.begin(), src.end()) != src.end() ? 1 : 0;
    }
    cudaError_t e = lsc::launch_restore(P, grid, stream);
    if (e != cudaSuccess) { cudaGetLastError(); return LSC_ERR_CUDA; }
    launches++;
  }
  if (done_event && cudaEventRecord((cudaEvent_t)done_event, stream) != cudaSuccess) return LSC_ERR_CUDA;
  rep.launches = launches;
  if (report) *report = rep;
  return rep.soft_cold ? LSC_SOFT_COLD : LSC_OK;
}

static int access_params(lsc_pool *p, int32_t layer, const int32_t *idx, int32_t n, lsc::AccessParams *a) {
  if (!p || n < 0) return LSC_ERR_INVALID_ARG;
  uint8_t *region;
  int rc = layer_base(p, layer, &region);
  if (rc != LSC_OK) return rc;
  if (n > 0 && !idx) return LSC_ERR_INVALID_ARG;
  rc = check_device(p);
  if (rc != LSC_OK) return rc;
  const lsc::Geom &g = p->g;
  memset(a, 0, sizeof(*a));
  a->layer = region;
  a->page = g.page;
  a->conv_bytes = g.conv_bytes;
  a->ssm_off = g.ssm_off;
  a->ssm_bytes = g.ssm_bytes;
  a->chunk_bytes = 32 << 10;
  a->num_slots = g.num_slots;
  a->n = n;
  a->conv_chunks = (int32_t)((g.conv_bytes + a->chunk_bytes - 1) / a->chunk_bytes);
  a->ssm_chunks = (int32_t)((g.ssm_bytes + a->chunk_bytes - 1) / a->chunk_bytes);
  a->idx = idx;
  a->status = g.status;
  return LSC_OK;
}

int lsc_gather(lsc_pool *p, int32_t layer, const int32_t *idx, const uint8_t *has_init, int32_t n,
               void *conv_dense, void *ssm_dense, void *stream) {
  lsc::TraceRange trace_("lsc_gather");
  lsc::AccessParams a;
  int rc = access_params(p, layer, idx, n, &a);
  if (rc != LSC_OK) return rc;
  if (n > 0 && (!conv_dense || !ssm_dense)) return LSC_ERR_INVALID_ARG;
  if (n == 0) return LSC_OK;
  a.has_init = has_init;
  a.conv_dense = (uint8_t *)conv_dense;
  a.ssm_dense = (uint8_t *)ssm_dense;
  if (lsc::launch_gather(a, p->num_sms, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  return LSC_OK;
}

int lsc_scatter(lsc_pool *p, int32_t layer, const int32_t *idx, int32_t n, const void *conv_dense,
                const void *ssm_dense, void *stream) {
  lsc::TraceRange trace_("lsc_scatter");
  lsc::AccessParams a;
  int rc = access_params(p, layer, idx, n, &a);
  if (rc != LSC_OK) return rc;
  if (n > 0 && (!conv_dense || !ssm_dense)) return LSC_ERR_INVALID_ARG;
  if (n == 0) return LSC_OK;
  a.conv_dense = (uint8_t *)conv_dense;
  a.ssm_dense = (uint8_t *)ssm_dense;
  if (lsc::launch_scatter(a, p->num_sms, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  return LSC_OK;
}

int lsc_gdn_decode(lsc_pool *p, int32_t layer, const lsc_gdn_decode_args *a, void *stream) {
  lsc::TraceRange trace_("lsc_gdn_decode");
  if (!p || !a) return LSC_ERR_INVALID_ARG;
  uint8_t *region;
  int rc = layer_base(p, layer, &region);
  if (rc != LSC_OK) return rc;
  const lsc::Geom &g = p->g;
  const int32_t Hk = a->num_k_heads;
  if (a->n < 0 || Hk <= 0 || g.Hv % Hk != 0 || g.conv_dim != 2 * Hk * g.dk + g.Hv * g.dv)
    return LSC_ERR_INVALID_ARG;
  if (a->n > 0 && (!a->idx || !a->x || !a->conv_weight || !a->alpha || !a->beta || !a->out))
    return LSC_ERR_INVALID_ARG;
  if ((a->flags & ~LSC_DECODE_EARLY_STATE) != 0) return LSC_ERR_INVALID_ARG;
  if (g.conv_dtype == LSC_F16 || g.ssm_dtype == LSC_F16) return LSC_ERR_UNSUPPORTED;
  if (g.conv_width > 8 || g.Hv / Hk > 8 || a->n > 65535) return LSC_ERR_UNSUPPORTED;
  if (!all_aligned({a->x, a->conv_weight}, (uintptr_t)esize(g.conv_dtype)) ||
      !all_aligned({a->idx, a->alpha, a->beta, a->out}, 4))
    return LSC_ERR_MISALIGNED;
  rc = check_device(p);
  if (rc != LSC_OK) return rc;
  if (a->n == 0) return LSC_OK;
  lsc::DecodeParams d{};
  d.layer = region;
  d.page = g.page;
  d.ssm_off = g.ssm_off;
  d.num_slots = g.num_slots;
  d.conv_dim = g.conv_dim;
  d.conv_width = g.conv_width;
  d.conv_bf16 = g.conv_dtype == LSC_BF16;
  d.Hk = Hk;
  d.Hv = g.Hv;
  d.dv = g.dv;
  d.group = g.Hv / Hk;
  d.n = a->n;
  d.idx = a->idx;
  d.has_init = a->has_init;
  d.x = a->x;
  d.w = a->conv_weight;
  d.alpha = a->alpha;
  d.beta = a->beta;
  d.out = a->out;
  d.status = g.status;
  // The vector conv path reads and writes 8-channel groups of the conv state,
  // x and the weights with 16-byte accesses: a work item's channels (q and k of
  // one q/k head, the v channels of its Hv/Hk heads) must be whole groups, and
  // every segment 16-byte aligned in start and length.
  const int64_t esc = g.conv_dtype == LSC_BF16 ? 2 : 4, W = g.conv_width;
  const int64_t units[] = {g.dk * (W - 1) * esc, (int64_t)g.dv * (W - 1) * esc, g.dk * esc, (int64_t)g.dv * esc,
                           (int64_t)g.conv_dim * esc, g.dk * W * esc, (int64_t)g.dv * W * esc};
  bool tma = ((uintptr_t)a->x % 16) == 0 && ((uintptr_t)a->conv_weight % 16) == 0 && g.dk % 8 == 0 &&
             ((int64_t)(g.Hv / Hk) * g.dv) % 8 == 0;
  for (int64_t u : units) tma = tma && (u % 16) == 0;
  d.conv_vec = tma ? 1 : 0;
  d.wait_limit_ns = fault("timeout0") ? 0 : kWaitLimitNs;
  d.drain_limit_ns = kWaitLimitNs;
  d.num_sms = p->num_sms;
  d.early_state = (a->flags & LSC_DECODE_EARLY_STATE) != 0;
  return lsc::launch_decode(d, g.dk, g.ssm_dtype, (cudaStream_t)stream);
}

int lsc_gdn_prefill_conv(lsc_pool *p, int32_t layer, const lsc_gdn_prefill_conv_args *a, void *stream) {
  lsc::TraceRange trace_("lsc_gdn_prefill_conv");
  if (!p || !a) return LSC_ERR_INVALID_ARG;
  uint8_t *region;
  int rc = layer_base(p, layer, &region);
  if (rc != LSC_OK) return rc;
  const lsc::Geom &g = p->g;
  const int32_t Hk = a->num_k_heads;
  if (a->n_seq < 0 || a->total_tokens < 0 || a->reserved != 0 || Hk <= 0 || g.Hv % Hk != 0 ||
      g.conv_dim != 2 * Hk * g.dk + g.Hv * g.dv)
    return LSC_ERR_INVALID_ARG;
  if (a->n_seq == 0 && a->total_tokens > 0) return LSC_ERR_INVALID_ARG;
  if (a->n_seq > 0 && (!a->idx || !a->cu_seqlens)) return LSC_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->x || !a->conv_weight || !a->q || !a->k || !a->v)) return LSC_ERR_INVALID_ARG;
  if (g.conv_dtype == LSC_F16) return LSC_ERR_UNSUPPORTED;
  if (g.conv_width > 8 || a->n_seq > 65535) return LSC_ERR_UNSUPPORTED;
  if (!all_aligned({a->x, a->conv_weight}, (uintptr_t)esize(g.conv_dtype)) ||
      !all_aligned({a->idx, a->cu_seqlens, a->q, a->k, a->v}, 4))
    return LSC_ERR_MISALIGNED;
  rc = check_device(p);
  if (rc != LSC_OK) return rc;
  if (a->n_seq == 0) return LSC_OK;
  lsc::PrefillConvParams d{};
  d.layer = region;
  d.page = g.page;
  d.num_slots = g.num_slots;
  d.conv_dim = g.conv_dim;
  d.conv_width = g.conv_width;
  d.conv_bf16 = g.conv_dtype == LSC_BF16;
  d.Hk = Hk;
  d.Hv = g.Hv;
  d.dk = g.dk;
  d.dv = g.dv;
  d.n_seq = a->n_seq;
  d.total_tokens = a->total_tokens;
  d.idx = a->idx;
  d.has_init = a->has_init;
  d.cu = a->cu_seqlens;
  d.x = a->x;
  d.w = a->conv_weight;
  d.q = a->q;
  d.k = a->k;
  d.v = a->v;
  d.status = g.status;
  // The fast path reads 8-channel groups of x, the weights and the conv state
  // with 16-byte loads, writes 8 outputs as two 16-byte stores, and reduces a
  // q/k head's sum of squares over dk / 8 consecutive lanes.
  const int tph = g.dk / 8;
  const bool pow2 = tph > 0 && tph <= 32 && (tph & (tph - 1)) == 0;
  const uintptr_t al = (uintptr_t)a->x | (uintptr_t)a->conv_weight | (uintptr_t)a->q | (uintptr_t)a->k |
                       (uintptr_t)a->v;
  d.vec = g.conv_dim % 8 == 0 && g.dk % 8 == 0 && g.dv % 8 == 0 && pow2 && (al % 16) == 0 ? 1 : 0;
  return lsc::launch_prefill_conv(d, (cudaStream_t)stream);
}

int lsc_gdn_recurrent(lsc_pool *p, int32_t layer, const lsc_gdn_recurrent_args *a, void *stream) {
  lsc::TraceRange trace_("lsc_gdn_recurrent");
  if (!p || !a) return LSC_ERR_INVALID_ARG;
  uint8_t *region;
  int rc = layer_base(p, layer, &region);
  if (rc != LSC_OK) return rc;
  const lsc::Geom &g = p->g;
  const int32_t Hk = a->num_k_heads;
  if (a->n_seq < 0 || a->total_tokens < 0 || Hk <= 0 || g.Hv % Hk != 0) return LSC_ERR_INVALID_ARG;
  if (a->algorithm < LSC_RECURRENT_AUTO || a->algorithm > LSC_RECURRENT_CHUNKED) return LSC_ERR_INVALID_ARG;
  if (a->n_seq > 0 && (!a->idx || !a->cu_seqlens)) return LSC_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->alpha || !a->beta || !a->out))
    return LSC_ERR_INVALID_ARG;
  if (((uintptr_t)a->q | (uintptr_t)a->k) & 15) return LSC_ERR_MISALIGNED;
  if (!all_aligned({a->idx, a->cu_seqlens, a->v, a->alpha, a->beta, a->out}, 4)) return LSC_ERR_MISALIGNED;
  if (g.ssm_dtype == LSC_F16) return LSC_ERR_UNSUPPORTED;
  if (a->n_seq > 65535) return LSC_ERR_UNSUPPORTED;
  // AUTO takes the chunked form on the tensor cores where it applies (head_k_dim
  // 128), the faster of the two there; the token kernels elsewhere
  const bool chunked = a->algorithm == LSC_RECURRENT_CHUNKED ||
                       (a->algorithm == LSC_RECURRENT_AUTO && g.dk == lsc::chunk::kDK);
  if (chunked && g.dk != lsc::chunk::kDK) return LSC_ERR_UNSUPPORTED;
  if (chunked && a->workspace != nullptr &&
      (((uintptr_t)a->workspace & 15) != 0 ||
       a->workspace_bytes < (size_t)lsc::chunk::workspace_bytes(a->total_tokens, a->n_seq, g.Hv)))
    return ((uintptr_t)a->workspace & 15) != 0 ? LSC_ERR_MISALIGNED : LSC_ERR_INVALID_ARG;
  rc = check_device(p);
  if (rc != LSC_OK) return rc;
  if (a->n_seq == 0) return LSC_OK;
  lsc::RecurrentParams r{};
  r.layer = region;
  r.page = g.page;
  r.ssm_off = g.ssm_off;
  r.num_slots = g.num_slots;
  r.Hk = Hk;
  r.Hv = g.Hv;
  r.dv = g.dv;
  r.group = g.Hv / Hk;
  r.n_seq = a->n_seq;
  r.total_tokens = a->total_tokens;
  r.idx = a->idx;
  r.has_init = a->has_init;
  r.cu = a->cu_seqlens;
  r.q = a->q;
  r.k = a->k;
  r.v = a->v;
  r.alpha = a->alpha;
  r.beta = a->beta;
  r.out = a->out;
  r.status = g.status;
  r.wait_limit_ns = fault("timeout0") ? 0 : kWaitLimitNs;
  r.drain_limit_ns = kWaitLimitNs;
  if (!chunked) return lsc::launch_recurrent(r, g.dk, g.ssm_dtype, (cudaStream_t)stream);
  // The chunked form: the preparation kernel writes every chunk's state-free
  // record into the workspace, the state kernel reads them, in stream order.
  const size_t need = (size_t)lsc::chunk::workspace_bytes(a->total_tokens, a->n_seq, g.Hv);
  void *ws = a->workspace;
  const bool own = ws == nullptr;
  if (own) {
    if (cudaMallocAsync(&ws, need, (cudaStream_t)stream) != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_NO_MEMORY;
    }
  }
  r.ws = static_cast<float *>(ws);
  rc = lsc::launch_chunk_prep(r, p->num_sms, (cudaStream_t)stream);
  if (rc == LSC_OK) rc = lsc::launch_recurrent_chunked_tc(r, g.dk, g.ssm_dtype, (cudaStream_t)stream);
  if (own && cudaFreeAsync(ws, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    if (rc == LSC_OK) rc = LSC_ERR_CUDA;
  }
  return rc;
}

int lsc_gdn_recurrent_workspace_bytes(const lsc_pool *p, const lsc_gdn_recurrent_args *a, size_t *bytes) {
  if (!p || !a || !bytes || a->n_seq < 0 || a->total_tokens < 0) return LSC_ERR_INVALID_ARG;
  const bool chunked = a->algorithm == LSC_RECURRENT_CHUNKED ||
                       (a->algorithm == LSC_RECURRENT_AUTO && p->g.dk == lsc::chunk::kDK);
  *bytes = chunked ? (size_t)lsc::chunk::workspace_bytes(a->total_tokens, a->n_seq, p->g.Hv) : 0;
  return LSC_OK;
}

}  // extern "C"
