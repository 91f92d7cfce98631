// lsc_kv.cu -- host side of the attention K/V block pool (include/lsc_kv.h):
// layout, views, and copy_prefix's validation and launch plans.  The copy
// kernel is kv_copy_kernel in lsc_copy.cu.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §3, §3.2, §3.4 (page-strided block views, separate K
//        and V views, the merged two-lane view)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", figure 2 (copy_prefix)
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "lsc_internal.h"
#include "lsc_kv.h"

struct lsc_kv_pool {
  lsc_kv_pool_desc d;
  int device = -1;  // -1: host-only pool (no GPU when created)
  int num_sms = 0;
  uint8_t *base = nullptr;
  bool owns_base = false;
  int64_t es = 0, row_bytes = 0, payload = 0, lane_bytes = 0, region_bytes = 0;
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

// [VA] §3: block stride = physical page size / element size, so the page must
// hold the logical block and divide by the element size; 16-byte vector copies
// add page % 16 == 0.
int describe(const lsc_kv_pool_desc *d, lsc_kv_pool *g) {
  if (!d || d->num_layers <= 0 || d->num_blocks <= 0 || d->block_tokens <= 0 || d->num_kv_heads <= 0 ||
      d->head_dim <= 0)
    return LSC_ERR_INVALID_ARG;
  const int es = esize(d->dtype);
  if (!es) return LSC_ERR_INVALID_ARG;
  g->d = *d;
  g->es = es;
  g->row_bytes = (int64_t)d->num_kv_heads * d->head_dim * es;
  g->payload = g->row_bytes * d->block_tokens;
  if (d->page_bytes < g->payload || d->page_bytes % es) return LSC_ERR_LAYOUT;
  if (d->page_bytes % 16) return LSC_ERR_MISALIGNED;
  g->lane_bytes = (int64_t)d->num_blocks * d->page_bytes;
  g->region_bytes = 2 * g->lane_bytes;
  return LSC_OK;
}

}  // namespace

extern "C" {

int lsc_kv_pool_required_bytes(const lsc_kv_pool_desc *desc, size_t *total_bytes) {
  if (!total_bytes) return LSC_ERR_INVALID_ARG;
  lsc_kv_pool g;
  const int rc = describe(desc, &g);
  if (rc != LSC_OK) return rc;
  *total_bytes = (size_t)g.d.num_layers * (size_t)g.region_bytes;
  return LSC_OK;
}

int lsc_kv_pool_create(const lsc_kv_pool_desc *desc, void *device_base, size_t base_bytes, lsc_kv_pool **out) {
  if (!out) return LSC_ERR_INVALID_ARG;
  *out = nullptr;
  lsc_kv_pool *p = new (std::nothrow) lsc_kv_pool();
  if (!p) return LSC_ERR_NO_MEMORY;
  int rc = describe(desc, p);
  if (rc != LSC_OK) {
    delete p;
    return rc;
  }
  const size_t need = (size_t)p->d.num_layers * (size_t)p->region_bytes;
  if (device_base) {
    if ((uintptr_t)device_base % 256) {
      delete p;
      return LSC_ERR_MISALIGNED;
    }
    if (base_bytes < need) {
      delete p;
      return LSC_ERR_NO_MEMORY;
    }
  }
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    if (!device_base) {
      delete p;
      return LSC_ERR_CUDA;
    }
    p->base = (uint8_t *)device_base;  // host-only: views, no copies
    *out = p;
    return LSC_OK;
  }
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return LSC_ERR_CUDA;
  }
  if (device_base) {
    p->base = (uint8_t *)device_base;
  } else {
    if (cudaMalloc(&p->base, need) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return LSC_ERR_NO_MEMORY;
    }
    p->owns_base = true;
  }
  *out = p;
  return LSC_OK;
}

int lsc_kv_pool_destroy(lsc_kv_pool *p) {
  if (!p) return LSC_ERR_INVALID_ARG;
  int rc = LSC_OK;
  if (p->owns_base) {
    if (cudaDeviceSynchronize() != cudaSuccess) rc = LSC_ERR_CUDA;
    cudaFree(p->base);
  }
  delete p;
  return rc;
}

int lsc_kv_pool_layer_view(const lsc_kv_pool *p, int32_t layer, lsc_kv_layer_view *v) {
  if (!p || !v) return LSC_ERR_INVALID_ARG;
  if (layer < 0 || layer >= p->d.num_layers) return LSC_ERR_OUT_OF_RANGE;
  std::memset(v, 0, sizeof(*v));
  uint8_t *region = p->base + (int64_t)layer * p->region_bytes;
  v->region = region;
  v->region_bytes = p->region_bytes;
  v->k = region;
  v->v = region + p->lane_bytes;
  v->shape[0] = p->d.num_blocks;
  v->shape[1] = p->d.block_tokens;
  v->shape[2] = p->d.num_kv_heads;
  v->shape[3] = p->d.head_dim;
  v->strides[0] = p->d.page_bytes / p->es;
  v->strides[1] = (int64_t)p->d.num_kv_heads * p->d.head_dim;
  v->strides[2] = p->d.head_dim;
  v->strides[3] = 1;
  v->lane_stride = p->lane_bytes / p->es;
  v->page_bytes = p->d.page_bytes;
  v->payload_bytes = p->payload;
  v->row_bytes = p->row_bytes;
  v->dtype = p->d.dtype;
  return LSC_OK;
}

int lsc_copy_prefix(lsc_kv_pool *p, const lsc_kv_copy_op *ops, int32_t n_ops, void *stream, void *done_event,
                    int64_t *bytes_copied) {
  lsc::TraceRange trace_("lsc_copy_prefix");
  if (!p || n_ops < 0 || (n_ops > 0 && !ops)) return LSC_ERR_INVALID_ARG;
  const int32_t B = p->d.num_blocks;
  // validate every copying op before enqueueing anything
  std::vector<int32_t> dst_owner;
  try {
    dst_owner.assign(B, -1);
  } catch (...) {
    return LSC_ERR_NO_MEMORY;
  }
  int64_t bytes = 0;
  int32_t n_copy = 0, last_copy = -1;
  for (int32_t r = 0; r < n_ops; ++r) {
    const lsc_kv_copy_op &o = ops[r];
    if (o.reserved != 0 || o.n_tokens < 0 || o.n_tokens > p->d.block_tokens) return LSC_ERR_INVALID_ARG;
    if (o.n_tokens == 0) continue;
    if (o.src_block < 0 || o.src_block >= B || o.dst_block < 0 || o.dst_block >= B) return LSC_ERR_OUT_OF_RANGE;
    if (dst_owner[o.dst_block] >= 0) return LSC_ERR_DUP_DST;
    dst_owner[o.dst_block] = r;
    bytes += (int64_t)o.n_tokens * p->row_bytes * 2 * p->d.num_layers;
    ++n_copy;
    last_copy = r;
  }
  for (int32_t r = 0; r < n_ops; ++r)
    if (ops[r].n_tokens > 0 && dst_owner[ops[r].src_block] >= 0) return LSC_ERR_SRC_IS_DST;
  if (p->device < 0) return LSC_ERR_CUDA;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  if (dev != p->device) return LSC_ERR_WRONG_DEVICE;
  cudaStream_t s = (cudaStream_t)stream;
  if (n_copy > 0) {
    static thread_local lsc::KvPlan plan;  // 30 KB: kept off the stack
    plan.base = p->base;
    plan.region_bytes = p->region_bytes;
    plan.lane_bytes = p->lane_bytes;
    plan.page = p->d.page_bytes;
    plan.row_bytes = p->row_bytes;
    plan.chunk_bytes = 32 << 10;
    plan.num_layers = p->d.num_layers;
    plan.chunks_per_op = (int32_t)((p->payload + plan.chunk_bytes - 1) / plan.chunk_bytes);
    plan.pad = 0;
    plan.n_ops = 0;
    for (int32_t r = 0; r < n_ops; ++r) {
      if (ops[r].n_tokens == 0) continue;
      plan.op[plan.n_ops++] = make_int3(ops[r].src_block, ops[r].dst_block, ops[r].n_tokens);
      if (plan.n_ops == lsc::kKvPlanMaxOps || r == last_copy) {
        if (lsc::launch_kv_copy(plan, p->num_sms, s) != cudaSuccess) {
          cudaGetLastError();
          return LSC_ERR_CUDA;
        }
        plan.n_ops = 0;
      }
    }
  }
  if (done_event && cudaEventRecord((cudaEvent_t)done_event, s) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_CUDA;
  }
  if (bytes_copied) *bytes_copied = bytes;
  return LSC_OK;
}

}  // extern "C"
