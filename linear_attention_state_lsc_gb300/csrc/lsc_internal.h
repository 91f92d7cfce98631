// lsc_internal.h -- shared between the host code and the kernels of liblsc.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "lsc.h"

namespace lsc {

// An NVTX range named after a public call, open for the call's duration, so
// that a timeline profiler shows each lsc_* call beside the kernels it
// enqueued.  NVTX v3 is header-only: without a profiler attached the push and
// pop return at once.
struct TraceRange {
  explicit TraceRange(const char *name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

// Launch with programmatic stream serialisation: the grid's CTAs may be placed
// while the previous kernel of the stream still runs; the kernel itself waits
// (griddepcontrol.wait) for that kernel's completion before any global access
// it does not own, and may let the next such kernel be placed early.
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<A &&>(args)...);
}

// ---- per-device launch state -------------------------------------------------
// A kernel's dynamic shared-memory limit (cudaFuncSetAttribute) and figures
// such as its occupancy belong to the device that is current at the call, and
// pools on different devices -- or several streams of one device -- may be
// driven from several host threads at once.  These records hold such values
// per device ordinal, read lock-free and written under a mutex.
constexpr int kMaxDevices = 64;

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`, once per device (the limit only ever grows, so a launch that
// checked it never sees it lowered by another thread).
class SmemLimit {
 public:
  cudaError_t ensure(const void *fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (set_[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (set_[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) set_[dev].store(bytes, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<int> set_[kMaxDevices] = {};
  std::mutex mu_;
};

// A positive integer computed once per device (on the device current at the
// first call from that device).  get() returns 0 when the current device
// cannot be read or `compute` returns a value below 1.
class PerDeviceInt {
 public:
  template <typename F>
  int get(F compute) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (dev < 0 || dev >= kMaxDevices) return compute(dev);
    int v = val_[dev].load(std::memory_order_acquire);
    if (v > 0) return v;
    std::lock_guard<std::mutex> lock(mu_);
    v = val_[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    v = compute(dev);
    if (v > 0) val_[dev].store(v, std::memory_order_release);
    return v > 0 ? v : 0;
  }

 private:
  std::atomic<int> val_[kMaxDevices] = {};
  std::mutex mu_;
};

// Byte geometry of one GDN layer region; the same for every GDN layer.
struct Geom {
  uint8_t *base;         // pool base (GDN layer g starts at base + g * region_bytes)
  int64_t page;          // physical page stride
  int64_t region_bytes;  // num_slots * page
  int64_t conv_bytes;    // conv view bytes, at page offset 0
  int64_t ssm_off;       // ssm view page offset (16 B aligned)
  int64_t ssm_bytes;
  int32_t num_slots;
  int32_t num_gdn;
  int32_t conv_dim, conv_width, conv_dtype;
  int32_t Hv, dv, dk, ssm_dtype;
  int32_t *status;       // device error word
};

// ---- restore -------------------------------------------------------------
// The whole plan travels as one by-value kernel parameter (<= 32764 bytes), so
// the call needs no staging buffer and no host sync.
constexpr int kPlanMaxHits = 2048;
constexpr int kPlanMaxHs = 3584;

struct RestorePlan {
  uint8_t *base;
  uint8_t *hs;             // device has_initial_state
  int64_t region_bytes;
  int64_t page;
  int64_t seg_off[2];      // copied byte ranges of a page
  int64_t seg_len[2];
  int64_t chunk_bytes;     // work-unit size
  int32_t seg_chunks[2];   // work units per segment
  int32_t chunks_per_slot;
  int32_t num_gdn;
  int32_t n_hits;
  int32_t n_hs;
  int32_t bulk;            // 1: copy through shared memory with 1-D TMA bulk copies
  int32_t src_reuse;       // 1: a source slot feeds several hits (its loads keep L2 priority)
  int32_t *status;         // device error word (bulk copies: a bounded wait gave up)
  int2 hit[kPlanMaxHits];  // (dst slot, src slot)
  int32_t hs_ops[kPlanMaxHs];  // (row << 1) | value
};
static_assert(sizeof(RestorePlan) <= 32000, "restore plan exceeds the kernel parameter limit");

cudaError_t launch_restore(const RestorePlan &plan, int grid, cudaStream_t stream);
int restore_grid(int num_sms);
int restore_bulk_grid(int num_sms);

// ---- gather / scatter ------------------------------------------------------
struct AccessParams {
  uint8_t *layer;          // region base of the GDN layer
  int64_t page, conv_bytes, ssm_off, ssm_bytes, chunk_bytes;
  int32_t num_slots, n, conv_chunks, ssm_chunks;
  const int32_t *idx;
  const uint8_t *has_init; // gather only, may be null
  uint8_t *conv_dense;
  uint8_t *ssm_dense;
  int32_t *status;
};
cudaError_t launch_gather(const AccessParams &p, int num_sms, cudaStream_t stream);
cudaError_t launch_scatter(const AccessParams &p, int num_sms, cudaStream_t stream);

// ---- GDN decode and recurrence ----------------------------------------------
struct DecodeParams {
  uint8_t *layer;
  int64_t page, ssm_off;
  int32_t num_slots, conv_dim, conv_width, conv_bf16;
  int32_t Hk, Hv, dv, group;
  int32_t n;
  const int32_t *idx;
  const uint8_t *has_init;
  const void *x;
  const void *w;
  const float *alpha, *beta;
  float *out;
  int32_t *status;
  int32_t conv_vec;         // conv segments 16-byte aligned: 8-channel vector path
  uint64_t wait_limit_ns;   // bound of each mbarrier wait (0: give up at once)
  uint64_t drain_limit_ns;  // bound of the wait for in-flight copies after a timeout
  int32_t num_sms;
  int32_t stages;           // set by the launcher: shared-memory ring depth
  int32_t early_state;      // LSC_DECODE_EARLY_STATE: rows and first state tiles read before griddep_wait()
};
// returns LSC_OK, LSC_ERR_UNSUPPORTED or LSC_ERR_CUDA
int launch_decode(const DecodeParams &p, int dk, int ssm_dtype, cudaStream_t stream);

struct RecurrentParams {
  uint8_t *layer;
  int64_t page, ssm_off;
  int32_t num_slots, Hk, Hv, dv, group, n_seq, total_tokens;
  const int32_t *idx;
  const uint8_t *has_init;
  const int32_t *cu;
  const float *q, *k, *v, *alpha, *beta;
  float *out;
  int32_t *status;
  uint64_t wait_limit_ns;   // bound of each mbarrier wait (tensor-core form; 0: give up at once)
  uint64_t drain_limit_ns;  // bound of the wait for issued MMAs after a timeout
  float *ws;                // chunked form: workspace records (lsc_chunk.h)
};
int launch_recurrent(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t stream);
// the token recurrence for head_k_dim 128 (lsc_rec128.cu)
int launch_recurrent128(const RecurrentParams &p, int ssm_dtype, cudaStream_t stream);
// the chunked evaluation on the tensor cores: head_k_dim 128, head_v_dim <= 128.
// launch_chunk_prep (lsc_chunk_prep.cu) writes the state-free records of
// every chunk to p.ws; launch_recurrent_chunked_tc (lsc_chunked_tc.cu), on
// the same stream after it, runs the state through the chunks.
int launch_chunk_prep(const RecurrentParams &p, int num_sms, cudaStream_t stream);
int launch_recurrent_chunked_tc(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t stream);

struct PrefillConvParams {
  uint8_t *layer;
  int64_t page;
  int32_t num_slots, conv_dim, conv_width, conv_bf16;
  int32_t Hk, Hv, dk, dv;
  int32_t n_seq, total_tokens;
  const int32_t *idx;
  const uint8_t *has_init;
  const int32_t *cu;
  const void *x;
  const void *w;
  float *q, *k, *v;
  int32_t *status;
  int32_t vec;  // fast path: 8-channel groups, q/k norm fused (see lsc_prefill.cu)
};
// returns LSC_OK, LSC_ERR_UNSUPPORTED or LSC_ERR_CUDA
int launch_prefill_conv(const PrefillConvParams &p, cudaStream_t stream);

// copy_prefix plan, passed by value (<= 32 KB of kernel parameters)
constexpr int kKvPlanMaxOps = 2560;
struct KvPlan {
  uint8_t *base;
  int64_t region_bytes;  // one attention layer: both lanes
  int64_t lane_bytes;    // num_blocks pages
  int64_t page, row_bytes, chunk_bytes;
  int32_t num_layers, n_ops, chunks_per_op, pad;
  int3 op[kKvPlanMaxOps];  // (src block, dst block, n_tokens > 0)
};
cudaError_t launch_kv_copy(const KvPlan &p, int num_sms, cudaStream_t stream);

}  // namespace lsc
