// lsc_copy.cu -- byte-moving kernels of liblsc: the persistent cross-layer
// restore, and the strided gather / scatter of slot state.
//
// Sources, cited by page title and section:
//   [XN] "Linear-State Prefix Cache 内部机制" §4.1, §4.3 (restore copy and the
//        has_initial_state write)
//   [VA] "非连续 KV Cache" §3 (page stride, padding skipped by stride), §4-§5
//        (gather_ssm_states / scatter_ssm_states_)
//
// All are HBM-bound copies.  They move whole 32 KiB chunks with 1-D TMA bulk
// copies (the restore, when the ranges allow) or 16-byte vectors with
// coalesced loads and streaming stores, never touch bytes outside the conv
// and ssm views of a page, and run as persistent grids sized from the SM
// count.
#include <cuda_runtime.h>

#include "lsc_internal.h"
#include "lsc_ptx.h"

namespace lsc {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;  // 16 B vectors in flight per thread

__device__ __forceinline__ void report(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// Every copy kernel is launched with programmatic stream serialisation
// (launch_pdl): its CTAs may be placed while the previous kernel of the stream
// runs, and wait here, before any global access, until that kernel has
// completed; then they let the next such kernel be placed early in turn.
__device__ __forceinline__ void pdl_enter() {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
}

// Block-cooperative copy of nvec 16 B vectors: every thread issues kUnroll
// loads before its stores, so a CTA keeps kThreads * kUnroll * 16 B in flight.
__device__ __forceinline__ void copy_vec16(uint4 *__restrict__ d, const uint4 *__restrict__ s,
                                           int64_t nvec) {
  int64_t i = threadIdx.x;
  const int64_t stride = blockDim.x;
  for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
    uint4 r[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) r[k] = __ldg(s + i + k * stride);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) __stcs(d + i + k * stride, r[k]);
  }
  for (; i < nvec; i += stride) __stcs(d + i, __ldg(s + i));
}

// Copy len bytes with the widest access the two addresses allow; the tail that
// does not fill a vector is copied byte by byte and stops exactly at len.
__device__ __forceinline__ void copy_span(uint8_t *dst, const uint8_t *src, int64_t len) {
  const uintptr_t a = (uintptr_t)dst | (uintptr_t)src;
  int64_t done = 0;
  if ((a & 15) == 0) {
    const int64_t nv = len >> 4;
    copy_vec16((uint4 *)dst, (const uint4 *)src, nv);
    done = nv << 4;
  } else if ((a & 3) == 0) {
    const int64_t nw = len >> 2;
    for (int64_t i = threadIdx.x; i < nw; i += blockDim.x)
      ((uint32_t *)dst)[i] = __ldg((const uint32_t *)src + i);
    done = nw << 2;
  }
  for (int64_t i = done + threadIdx.x; i < len; i += blockDim.x) dst[i] = src[i];
}

__device__ __forceinline__ void zero_span(uint8_t *dst, int64_t len) {
  int64_t done = 0;
  if (((uintptr_t)dst & 15) == 0) {
    const int64_t nv = len >> 4;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int64_t i = threadIdx.x; i < nv; i += blockDim.x) __stcs((uint4 *)dst + i, z);
    done = nv << 4;
  }
  for (int64_t i = done + threadIdx.x; i < len; i += blockDim.x) dst[i] = 0;
}

// Persistent restore: one launch covers every (hit row, GDN layer, chunk) work
// unit of the plan, plus the has_initial_state writes of the plan's rows.
// Consecutive units are consecutive chunks of one page, so at any moment the
// grid streams a contiguous stretch of each source page.
__global__ void __launch_bounds__(kThreads) restore_kernel(const __grid_constant__ RestorePlan p) {
  pdl_enter();
  const int gthreads = gridDim.x * blockDim.x;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < p.n_hs; j += gthreads) {
    const int32_t e = p.hs_ops[j];
    p.hs[e >> 1] = (uint8_t)(e & 1);
  }
  const int64_t per_hit = (int64_t)p.num_gdn * p.chunks_per_slot;
  const int64_t total = (int64_t)p.n_hits * per_hit;
  for (int64_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int h = (int)(u / per_hit);
    const int64_t rem = u - (int64_t)h * per_hit;
    const int g = (int)(rem / p.chunks_per_slot);
    int c = (int)(rem - (int64_t)g * p.chunks_per_slot);
    const int s = c >= p.seg_chunks[0] ? 1 : 0;
    if (s) c -= p.seg_chunks[0];
    const int64_t off = p.seg_off[s] + (int64_t)c * p.chunk_bytes;
    const int64_t left = p.seg_len[s] - (int64_t)c * p.chunk_bytes;
    const int64_t len = left < p.chunk_bytes ? left : p.chunk_bytes;
    uint8_t *layer = p.base + (int64_t)g * p.region_bytes;
    const int2 hs = p.hit[h];
    copy_span(layer + (int64_t)hs.x * p.page + off, layer + (int64_t)hs.y * p.page + off, len);
  }
}

// The same restore through shared memory with 1-D TMA bulk copies, the
// default when every copied range is 16-byte aligned in offset and length:
// one warp per CTA, two CTAs per SM, a ring of kBulkStages 32 KiB stages.  Its
// thread 0 keeps kBulkStages - 1 loads in flight: unit k is stored from its
// stage once its load has landed, and the load of unit k + kBulkStages - 1
// reuses the stage of unit k - 1 once that unit's store has read it.  Needs
// every copied range 16-byte aligned in offset and length (the host checks).
constexpr int kBulkStages = 3;
constexpr uint32_t kBulkChunk = 32 << 10;
constexpr uint64_t kBulkWaitNs = 1000000000ull;

__global__ void __launch_bounds__(32) restore_bulk_kernel(const __grid_constant__ RestorePlan p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kBulkStages];
  pdl_enter();
  const int gthreads = gridDim.x * blockDim.x;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < p.n_hs; j += gthreads) {
    const int32_t e = p.hs_ops[j];
    p.hs[e >> 1] = (uint8_t)(e & 1);
  }
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kBulkStages; ++s) mbar_init(&full[s], 1);
  fence_mbar_init();
  // Stores and single-use sources are streamed past L2 (evict first); a
  // source slot that feeds several hits (a hot checkpoint) keeps the default
  // priority, so its later reads hit L2 (the c3 storm: 4.61 -> 4.47 ms; with
  // every source used once the default priority cost 0.6 %).
  const uint64_t pol = l2_evict_first_policy();
  const uint64_t pol_ld = p.src_reuse ? l2_evict_normal_policy() : pol;
  const int64_t per_hit = (int64_t)p.num_gdn * p.chunks_per_slot;
  const int64_t total = (int64_t)p.n_hits * per_hit;
  const int64_t n = total > blockIdx.x ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  // unit k of this CTA -> (dst, src, len)
  auto unit = [&](int64_t k, uint8_t *&dst, const uint8_t *&src, uint32_t &len) {
    const int64_t u = blockIdx.x + k * gridDim.x;
    const int h = (int)(u / per_hit);
    const int64_t rem = u - (int64_t)h * per_hit;
    const int g = (int)(rem / p.chunks_per_slot);
    int c = (int)(rem - (int64_t)g * p.chunks_per_slot);
    const int s = c >= p.seg_chunks[0] ? 1 : 0;
    if (s) c -= p.seg_chunks[0];
    const int64_t off = p.seg_off[s] + (int64_t)c * p.chunk_bytes;
    const int64_t left = p.seg_len[s] - (int64_t)c * p.chunk_bytes;
    len = (uint32_t)(left < p.chunk_bytes ? left : p.chunk_bytes);
    uint8_t *layer = p.base + (int64_t)g * p.region_bytes;
    const int2 hs = p.hit[h];
    dst = layer + (int64_t)hs.x * p.page + off;
    src = layer + (int64_t)hs.y * p.page + off;
  };
  auto load = [&](int64_t k) {
    uint8_t *dst;
    const uint8_t *src;
    uint32_t len;
    unit(k, dst, src, len);
    const int st = (int)(k % kBulkStages);
    mbar_arrive_expect_tx(&full[st], len);
    bulk_g2s(ring + (size_t)st * kBulkChunk, src, len, &full[st], pol_ld);
  };
  for (int64_t k = 0; k < kBulkStages - 1 && k < n; ++k) load(k);
  for (int64_t k = 0; k < n; ++k) {
    const int st = (int)(k % kBulkStages);
    if (!mbar_wait_bounded(&full[st], (uint32_t)((k / kBulkStages) & 1), kBulkWaitNs)) {
      report(p.status, LSC_ERR_DEV_TIMEOUT);
      break;
    }
    uint8_t *dst;
    const uint8_t *src;
    uint32_t len;
    unit(k, dst, src, len);
    bulk_s2g(dst, ring + (size_t)st * kBulkChunk, len, pol);
    bulk_commit();
    if (k + kBulkStages - 1 < n) {
      bulk_wait_read_one();  // unit k - 1's store has read its stage
      load(k + kBulkStages - 1);
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // every store complete before exit
}

// copy_prefix: unit = (op, attention layer, lane, chunk of the op's rows);
// the rows [0, n) of a block are one contiguous span of n * row_bytes bytes.
__global__ void __launch_bounds__(kThreads) kv_copy_kernel(const __grid_constant__ KvPlan p) {
  pdl_enter();
  const int64_t per_op = (int64_t)p.num_layers * 2 * p.chunks_per_op;
  const int64_t total = (int64_t)p.n_ops * per_op;
  for (int64_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int o = (int)(u / per_op);
    int64_t rem = u - (int64_t)o * per_op;
    const int l = (int)(rem / (2 * p.chunks_per_op));
    rem -= (int64_t)l * 2 * p.chunks_per_op;
    const int lane = (int)(rem / p.chunks_per_op);
    const int c = (int)(rem - (int64_t)lane * p.chunks_per_op);
    const int3 op = p.op[o];
    const int64_t span = (int64_t)op.z * p.row_bytes;
    const int64_t off = (int64_t)c * p.chunk_bytes;
    if (off >= span) continue;  // a partial block has fewer chunks
    const int64_t len = span - off < p.chunk_bytes ? span - off : p.chunk_bytes;
    uint8_t *lane_base = p.base + (int64_t)l * p.region_bytes + (int64_t)lane * p.lane_bytes;
    copy_span(lane_base + (int64_t)op.y * p.page + off, lane_base + (int64_t)op.x * p.page + off, len);
  }
}

// Gather: unit = (row, chunk of the conv view or of the ssm view).
__global__ void __launch_bounds__(kThreads) gather_kernel(const __grid_constant__ AccessParams p) {
  pdl_enter();
  const int cps = p.conv_chunks + p.ssm_chunks;
  const int64_t total = (int64_t)p.n * cps;
  for (int64_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int i = (int)(u / cps);
    const int c = (int)(u - (int64_t)i * cps);
    const int32_t slot = p.idx[i];
    bool warm = slot >= 0 && (p.has_init == nullptr || p.has_init[i] != 0);
    if (slot >= p.num_slots) {
      warm = false;
      if (threadIdx.x == 0 && c == 0) report(p.status, LSC_ERR_OUT_OF_RANGE);
    }
    int64_t off, len, page_off;
    uint8_t *dst;
    if (c < p.conv_chunks) {
      off = (int64_t)c * p.chunk_bytes;
      len = p.conv_bytes - off < p.chunk_bytes ? p.conv_bytes - off : p.chunk_bytes;
      dst = p.conv_dense + (int64_t)i * p.conv_bytes + off;
      page_off = off;
    } else {
      off = (int64_t)(c - p.conv_chunks) * p.chunk_bytes;
      len = p.ssm_bytes - off < p.chunk_bytes ? p.ssm_bytes - off : p.chunk_bytes;
      dst = p.ssm_dense + (int64_t)i * p.ssm_bytes + off;
      page_off = p.ssm_off + off;
    }
    if (warm) copy_span(dst, p.layer + (int64_t)slot * p.page + page_off, len);
    else zero_span(dst, len);
  }
}

// Scatter: the inverse; negative or out-of-range indices write nothing.
__global__ void __launch_bounds__(kThreads) scatter_kernel(const __grid_constant__ AccessParams p) {
  pdl_enter();
  const int cps = p.conv_chunks + p.ssm_chunks;
  const int64_t total = (int64_t)p.n * cps;
  for (int64_t u = blockIdx.x; u < total; u += gridDim.x) {
    const int i = (int)(u / cps);
    const int c = (int)(u - (int64_t)i * cps);
    const int32_t slot = p.idx[i];
    if (slot < 0) continue;
    if (slot >= p.num_slots) {
      if (threadIdx.x == 0 && c == 0) report(p.status, LSC_ERR_OUT_OF_RANGE);
      continue;
    }
    int64_t off, len, page_off;
    const uint8_t *src;
    if (c < p.conv_chunks) {
      off = (int64_t)c * p.chunk_bytes;
      len = p.conv_bytes - off < p.chunk_bytes ? p.conv_bytes - off : p.chunk_bytes;
      src = p.conv_dense + (int64_t)i * p.conv_bytes + off;
      page_off = off;
    } else {
      off = (int64_t)(c - p.conv_chunks) * p.chunk_bytes;
      len = p.ssm_bytes - off < p.chunk_bytes ? p.ssm_bytes - off : p.chunk_bytes;
      src = p.ssm_dense + (int64_t)i * p.ssm_bytes + off;
      page_off = p.ssm_off + off;
    }
    copy_span(p.layer + (int64_t)slot * p.page + page_off, src, len);
  }
}

int blocks_per_sm(const void *kernel) {
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess || b < 1) {
    cudaGetLastError();
    b = 1;
  }
  return b;
}

// resident CTAs per SM of each copy kernel, per device
PerDeviceInt g_bps_restore, g_bps_gather, g_bps_scatter, g_bps_kv;

int grid_for(const void *kernel, int num_sms, int64_t units) {
  PerDeviceInt &rec = kernel == (const void *)restore_kernel  ? g_bps_restore
                      : kernel == (const void *)gather_kernel ? g_bps_gather
                      : kernel == (const void *)kv_copy_kernel ? g_bps_kv
                                                               : g_bps_scatter;
  int bps = rec.get([kernel](int) { return blocks_per_sm(kernel); });
  if (bps < 1) bps = 1;
  int64_t g = (int64_t)num_sms * bps;
  if (units < g) g = units;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

int restore_grid(int num_sms) { return grid_for((const void *)restore_kernel, num_sms, 1LL << 40); }
int restore_bulk_grid(int num_sms) { return 2 * num_sms; }

SmemLimit g_bulk_smem;

cudaError_t launch_restore(const RestorePlan &plan, int grid, cudaStream_t stream) {
  cudaError_t e;
  if (plan.bulk) {
    const int smem = kBulkStages * (int)kBulkChunk;
    e = g_bulk_smem.ensure((const void *)restore_bulk_kernel, smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(restore_bulk_kernel, grid, 32, smem, stream, plan);
  } else {
    e = launch_pdl(restore_kernel, grid, kThreads, 0, stream, plan);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_gather(const AccessParams &p, int num_sms, cudaStream_t stream) {
  const int64_t units = (int64_t)p.n * (p.conv_chunks + p.ssm_chunks);
  const cudaError_t e = launch_pdl(gather_kernel, grid_for((const void *)gather_kernel, num_sms, units), kThreads, 0,
                                   stream, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_kv_copy(const KvPlan &p, int num_sms, cudaStream_t stream) {
  const int64_t units = (int64_t)p.n_ops * p.num_layers * 2 * p.chunks_per_op;
  if (units == 0) return cudaSuccess;
  const cudaError_t e = launch_pdl(kv_copy_kernel, grid_for((const void *)kv_copy_kernel, num_sms, units), kThreads,
                                   0, stream, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_scatter(const AccessParams &p, int num_sms, cudaStream_t stream) {
  const int64_t units = (int64_t)p.n * (p.conv_chunks + p.ssm_chunks);
  const cudaError_t e = launch_pdl(scatter_kernel, grid_for((const void *)scatter_kernel, num_sms, units), kThreads,
                                   0, stream, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace lsc
