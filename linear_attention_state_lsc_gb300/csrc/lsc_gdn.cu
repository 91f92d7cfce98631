// lsc_gdn.cu -- GDN kernels of liblsc: the fused decode step (strided gather ->
// causal_conv1d_update -> gated delta rule -> in-place scatter) and the
// token-by-token recurrence of a resumed prefill.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §5 (state indices -> strided state -> gather -> FLA
//        kernel -> scatter), §6 (causal_conv1d_update, recurrent_gated_delta_rule)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with q)
//
// The delta rule S' = a S (I - b k k^T) + b v k^T is applied row by row:
// for row r of S,  u_r = S_r . k,  d_r = b (v_r - a u_r),  S'_r = a S_r + d_r k,
// and o_r = S'_r . q = a (S_r . q) + d_r (k . q).  Each row needs only its own
// elements and the broadcast vectors k, q, so the state streams through
// registers once: one HBM read and one HBM write per element.  No tensor cores:
// a decode token is a rank-1 update, about 2 flops per state byte.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lsc_internal.h"

namespace lsc {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kMaxDv = 128;
constexpr int kMaxTaps = 8;

__device__ __forceinline__ void report(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// Conv-side element access (conv dtype is f32 or bf16, chosen at run time).
__device__ __forceinline__ float ld_conv(const void *base, int64_t i, bool bf16) {
  return bf16 ? bf16_bits_to_float(((const uint16_t *)base)[i]) : ((const float *)base)[i];
}
__device__ __forceinline__ void st_conv(void *base, int64_t i, float v, bool bf16) {
  if (bf16) ((uint16_t *)base)[i] = float_to_bf16_bits(v);
  else ((float *)base)[i] = v;
}

// 16-byte vectors of state elements <-> floats.
template <typename TS> struct StateVec;
template <> struct StateVec<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <> struct StateVec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 pack(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);  // .x = low half
      w[k] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Fused decode.  Grid (Hv, n); a cluster spans the `group` v heads that share
// one q/k head, so every CTA of a cluster works on the same row.  CTA (h, i):
//  1. issues the loads of its head's [dv x DK] state slice into registers (they
//     complete while the conv runs);
//  2. runs the conv update for the q and k channels of head group g and the v
//     channels of head h, keeping y in shared memory; v channels' new conv state
//     is written at once (this CTA owns them);
//  3. waits on the cluster barrier -- every CTA of the cluster has now read the
//     shared q/k channels' old conv state -- after which cluster rank 0 writes
//     their new state;
//  4. L2-normalises q and k, then updates its state rows and writes o.
// Thread layout: TPR threads per state row, NV 16-byte vectors per thread;
// vector j of a thread is column vector j*TPR + lane_in_row, so a warp's loads
// use whole 32-byte sectors.
template <int DK, typename TS, int PASSES>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int EPV = StateVec<TS>::kElems;
  constexpr int VPR = DK / EPV;
  constexpr int NV = VPR < 8 ? VPR : 8;
  constexpr int TPR = VPR / NV;
  constexpr int RPP = kDecodeThreads / TPR;
  static_assert(VPR % NV == 0 && TPR >= 1 && TPR <= 32, "state row layout");

  __shared__ __align__(16) float ys[2 * DK + kMaxDv];
  __shared__ float qk_stash[2 * DK * (kMaxTaps - 1)];
  __shared__ float red[3][kDecodeThreads / 32];

  const int tid = threadIdx.x;
  const int h = blockIdx.x, i = blockIdx.y;
  const int g = h / p.group;
  const bool rank0 = (h % p.group) == 0;
  const int32_t slot = p.idx[i];
  const bool bad = slot >= p.num_slots;
  const bool valid = slot >= 0 && !bad;
  const bool warm = valid && (p.has_init == nullptr || p.has_init[i] != 0);
  if (bad && tid == 0 && rank0) report(p.status, LSC_ERR_OUT_OF_RANGE);

  uint8_t *page = valid ? p.layer + (int64_t)slot * p.page : nullptr;
  TS *S = valid ? (TS *)(page + p.ssm_off) + (int64_t)h * p.dv * DK : nullptr;
  const int r0 = tid / TPR, lr = tid % TPR;

  // 1. state prefetch
  uint4 sreg[PASSES][NV];
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = r0 + ps * RPP;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (warm && r < p.dv) sreg[ps][j] = *(const uint4 *)(S + (int64_t)r * DK + (j * TPR + lr) * EPV);
      else sreg[ps][j] = make_uint4(0, 0, 0, 0);
    }
  }

  // 2. causal conv1d update of this CTA's channels
  const int C = p.conv_dim, W = p.conv_width;
  const bool cbf = p.conv_bf16 != 0;
  const int nch = 2 * DK + p.dv;
  for (int cl = tid; cl < nch; cl += kDecodeThreads) {
    const int c = cl < DK ? g * DK + cl
                          : (cl < 2 * DK ? p.Hk * DK + g * DK + (cl - DK) : 2 * p.Hk * DK + h * p.dv + (cl - 2 * DK));
    float win[kMaxTaps];
    for (int j = 0; j < W - 1; ++j) win[j] = warm ? ld_conv(page, (int64_t)c * (W - 1) + j, cbf) : 0.f;
    win[W - 1] = ld_conv(p.x, (int64_t)i * C + c, cbf);
    float z = 0.f;
    for (int j = 0; j < W; ++j) z = fmaf(ld_conv(p.w, (int64_t)c * W + j, cbf), win[j], z);
    ys[cl] = z / (1.f + expf(-z));  // SiLU
    if (valid) {
      if (cl >= 2 * DK) {
        for (int j = 0; j < W - 1; ++j) st_conv(page, (int64_t)c * (W - 1) + j, win[j + 1], cbf);
      } else {
        for (int j = 0; j < W - 1; ++j) qk_stash[cl * (W - 1) + j] = win[j + 1];
      }
    }
  }

  // 3. every CTA of the cluster has read the shared q/k conv state
  cluster_sync_all();
  if (valid && rank0) {
    for (int cl = tid; cl < 2 * DK; cl += kDecodeThreads) {
      const int c = cl < DK ? g * DK + cl : p.Hk * DK + g * DK + (cl - DK);
      for (int j = 0; j < W - 1; ++j) st_conv(page, (int64_t)c * (W - 1) + j, qk_stash[cl * (W - 1) + j], cbf);
    }
  }

  // 4a. L2 norms of q and k, and k . q
  float sq = 0.f, sk = 0.f, sqk = 0.f;
  for (int c = tid; c < DK; c += kDecodeThreads) {
    const float a = ys[c], b = ys[DK + c];
    sq = fmaf(a, a, sq);
    sk = fmaf(b, b, sk);
    sqk = fmaf(a, b, sqk);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, m);
    sk += __shfl_xor_sync(0xffffffffu, sk, m);
    sqk += __shfl_xor_sync(0xffffffffu, sqk, m);
  }
  if ((tid & 31) == 0) {
    red[0][tid >> 5] = sq;
    red[1][tid >> 5] = sk;
    red[2][tid >> 5] = sqk;
  }
  __syncthreads();
  sq = sk = sqk = 0.f;
#pragma unroll
  for (int w = 0; w < kDecodeThreads / 32; ++w) {
    sq += red[0][w];
    sk += red[1][w];
    sqk += red[2][w];
  }
  const float inv_q = 1.f / sqrtf(sq + 1e-6f);
  const float inv_k = 1.f / sqrtf(sk + 1e-6f);
  const float kq = sqk * inv_q * inv_k;
  for (int c = tid; c < 2 * DK; c += kDecodeThreads) ys[c] *= c < DK ? inv_q : inv_k;
  __syncthreads();

  // 4b. delta rule on the register-resident rows
  const float a = valid ? p.alpha[(int64_t)i * p.Hv + h] : 0.f;
  const float b = valid ? p.beta[(int64_t)i * p.Hv + h] : 0.f;
  const float *qs = ys, *ks = ys + DK;
#pragma unroll
  for (int ps = 0; ps < PASSES; ++ps) {
    const int r = r0 + ps * RPP;
    const bool rv = r < p.dv;
    float u = 0.f, wq = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float s[EPV];
      StateVec<TS>::unpack(sreg[ps][j], s);
      const int c0 = (j * TPR + lr) * EPV;
#pragma unroll
      for (int e = 0; e < EPV; e += 4) {
        const float4 k4 = *(const float4 *)(ks + c0 + e);
        const float4 q4 = *(const float4 *)(qs + c0 + e);
        u = fmaf(s[e], k4.x, u); u = fmaf(s[e + 1], k4.y, u); u = fmaf(s[e + 2], k4.z, u); u = fmaf(s[e + 3], k4.w, u);
        wq = fmaf(s[e], q4.x, wq); wq = fmaf(s[e + 1], q4.y, wq); wq = fmaf(s[e + 2], q4.z, wq); wq = fmaf(s[e + 3], q4.w, wq);
      }
    }
#pragma unroll
    for (int m = TPR / 2; m >= 1; m >>= 1) {
      u += __shfl_xor_sync(0xffffffffu, u, m);
      wq += __shfl_xor_sync(0xffffffffu, wq, m);
    }
    const float vr = rv ? ys[2 * DK + r] : 0.f;
    const float d = b * (vr - a * u);
    const float o = fmaf(a, wq, d * kq);
    if (valid && rv) {
      TS *row = S + (int64_t)r * DK;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        float s[EPV];
        StateVec<TS>::unpack(sreg[ps][j], s);
        const int c0 = (j * TPR + lr) * EPV;
#pragma unroll
        for (int e = 0; e < EPV; ++e) s[e] = fmaf(a, s[e], d * ks[c0 + e]);
        __stcs((uint4 *)(row + c0), StateVec<TS>::pack(s));
      }
    }
    if (rv && lr == 0) p.out[((int64_t)i * p.Hv + h) * p.dv + r] = valid ? o : 0.f;
  }
}

template <int DK, typename TS, int PASSES>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hv, p.n, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.group;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<DK, TS, PASSES>, p);
}

template <int DK, typename TS>
int dispatch_decode_passes(const DecodeParams &p, cudaStream_t s) {
  constexpr int EPV = StateVec<TS>::kElems;
  constexpr int VPR = DK / EPV;
  constexpr int NV = VPR < 8 ? VPR : 8;
  constexpr int RPP = kDecodeThreads / (VPR / NV);
  const int passes = (p.dv + RPP - 1) / RPP;
  cudaError_t e;
  if (passes == 1) e = launch_decode_t<DK, TS, 1>(p, s);
  else if constexpr (RPP * 2 >= kMaxDv && RPP < kMaxDv) {
    if (passes == 2) e = launch_decode_t<DK, TS, 2>(p, s);
    else return LSC_ERR_UNSUPPORTED;
  } else return LSC_ERR_UNSUPPORTED;
  if (e != cudaSuccess) { cudaGetLastError(); return LSC_ERR_CUDA; }
  return LSC_OK;
}

// ---------------------------------------------------------------------------
// Token-by-token recurrence.  Grid (Hv, n_seq), one CTA per (sequence, v head);
// row r of the head's state lives in the registers of TPR threads (CPT columns
// each) for the whole sequence.  Tokens are staged in shared memory TT at a
// time; k . q of each token is computed once per tile.
constexpr int kTileTokens = 16;

template <int DK, typename TS>
__global__ void __launch_bounds__(512, 1) recurrent_kernel(const __grid_constant__ RecurrentParams p) {
  constexpr int CPT = DK < 32 ? DK : 32;
  constexpr int TPR = DK / CPT;
  constexpr int NV4 = CPT / 4;
  constexpr int TT = kTileTokens;
  __shared__ __align__(16) float sq[TT][DK];
  __shared__ __align__(16) float sk[TT][DK];
  __shared__ float sv[TT][kMaxDv];
  __shared__ float sa[TT], sb[TT], skq[TT];

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int h = blockIdx.x, i = blockIdx.y;
  const int g = h / p.group;
  const int32_t slot = p.idx[i];
  const bool bad = slot >= p.num_slots;
  const bool valid = slot >= 0 && !bad;
  const bool warm = valid && (p.has_init == nullptr || p.has_init[i] != 0);
  const int t0 = p.cu[i], t1 = p.cu[i + 1];
  if (bad && tid == 0 && h == 0) report(p.status, LSC_ERR_OUT_OF_RANGE);
  if (t0 < 0 || t1 < t0 || t1 > p.total_tokens) {  // inconsistent cu_seqlens: touch nothing
    if (tid == 0 && h == 0) report(p.status, LSC_ERR_INVALID_ARG);
    return;
  }
  const int dv = p.dv;
  const int r = tid / TPR, lr = tid % TPR;
  const bool rv = r < dv;

  if (!valid) {  // uniform over the CTA
    for (int64_t e = tid; e < (int64_t)(t1 - t0) * dv; e += nthr) {
      const int64_t t = t0 + e / dv;
      p.out[(t * p.Hv + h) * dv + e % dv] = 0.f;
    }
    return;
  }

  TS *Srow = (TS *)(p.layer + (int64_t)slot * p.page + p.ssm_off) + ((int64_t)h * dv + (rv ? r : 0)) * DK;
  float S[CPT];
#pragma unroll
  for (int j = 0; j < NV4; ++j) {
    const int c0 = (j * TPR + lr) * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = 0.f;
      if (warm && rv) {
        if constexpr (sizeof(TS) == 4) v = ((const float *)Srow)[c0 + e];
        else v = bf16_bits_to_float(((const uint16_t *)Srow)[c0 + e]);
      }
      S[j * 4 + e] = v;
    }
  }

  const int nwarps = (nthr + 31) >> 5, warp = tid >> 5, lane = tid & 31;
  for (int tb = t0; tb < t1; tb += TT) {
    const int nt = t1 - tb < TT ? t1 - tb : TT;
    __syncthreads();
    for (int e = tid; e < nt * (DK / 4); e += nthr) {
      const int tt = e / (DK / 4), c4 = e % (DK / 4);
      const int64_t src = ((int64_t)(tb + tt) * p.Hk + g) * DK + c4 * 4;
      *(float4 *)&sq[tt][c4 * 4] = *(const float4 *)(p.q + src);
      *(float4 *)&sk[tt][c4 * 4] = *(const float4 *)(p.k + src);
    }
    for (int e = tid; e < nt * dv; e += nthr) {
      const int tt = e / dv, c = e % dv;
      sv[tt][c] = p.v[((int64_t)(tb + tt) * p.Hv + h) * dv + c];
    }
    if (tid < nt) {
      sa[tid] = p.alpha[(int64_t)(tb + tid) * p.Hv + h];
      sb[tid] = p.beta[(int64_t)(tb + tid) * p.Hv + h];
    }
    __syncthreads();
    for (int tt = warp; tt < nt; tt += nwarps) {
      float acc = 0.f;
      for (int c = lane; c < DK; c += 32) acc = fmaf(sq[tt][c], sk[tt][c], acc);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      if (lane == 0) skq[tt] = acc;
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      // four partial sums per dot product keep the FMA chains short
      float u4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NV4; ++j) {
        const int c0 = (j * TPR + lr) * 4;
        const float4 k4 = *(const float4 *)&sk[tt][c0];
        const float4 q4 = *(const float4 *)&sq[tt][c0];
        u4[0] = fmaf(S[j * 4], k4.x, u4[0]); u4[1] = fmaf(S[j * 4 + 1], k4.y, u4[1]);
        u4[2] = fmaf(S[j * 4 + 2], k4.z, u4[2]); u4[3] = fmaf(S[j * 4 + 3], k4.w, u4[3]);
        w4[0] = fmaf(S[j * 4], q4.x, w4[0]); w4[1] = fmaf(S[j * 4 + 1], q4.y, w4[1]);
        w4[2] = fmaf(S[j * 4 + 2], q4.z, w4[2]); w4[3] = fmaf(S[j * 4 + 3], q4.w, w4[3]);
      }
      float u = (u4[0] + u4[1]) + (u4[2] + u4[3]);
      float wq = (w4[0] + w4[1]) + (w4[2] + w4[3]);
#pragma unroll
      for (int m = TPR / 2; m >= 1; m >>= 1) {
        u += __shfl_xor_sync(0xffffffffu, u, m);
        wq += __shfl_xor_sync(0xffffffffu, wq, m);
      }
      const float a = sa[tt], b = sb[tt];
      const float vr = rv ? sv[tt][r] : 0.f;
      const float d = b * (vr - a * u);
#pragma unroll
      for (int j = 0; j < NV4; ++j) {
        const int c0 = (j * TPR + lr) * 4;
        const float4 k4 = *(const float4 *)&sk[tt][c0];
        S[j * 4] = fmaf(a, S[j * 4], d * k4.x);
        S[j * 4 + 1] = fmaf(a, S[j * 4 + 1], d * k4.y);
        S[j * 4 + 2] = fmaf(a, S[j * 4 + 2], d * k4.z);
        S[j * 4 + 3] = fmaf(a, S[j * 4 + 3], d * k4.w);
      }
      if (rv && lr == 0) p.out[((int64_t)(tb + tt) * p.Hv + h) * dv + r] = fmaf(a, wq, d * skq[tt]);
    }
  }

  if (rv) {
#pragma unroll
    for (int j = 0; j < NV4; ++j) {
      const int c0 = (j * TPR + lr) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (sizeof(TS) == 4) ((float *)Srow)[c0 + e] = S[j * 4 + e];
        else ((uint16_t *)Srow)[c0 + e] = float_to_bf16_bits(S[j * 4 + e]);
      }
    }
  }
}

template <int DK, typename TS>
int launch_recurrent_t(const RecurrentParams &p, cudaStream_t s) {
  constexpr int CPT = DK < 32 ? DK : 32;
  constexpr int TPR = DK / CPT;
  int threads = (p.dv * TPR + 31) / 32 * 32;
  if (threads > 512) return LSC_ERR_UNSUPPORTED;
  recurrent_kernel<DK, TS><<<dim3(p.Hv, p.n_seq, 1), threads, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace

int launch_decode(const DecodeParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (p.dv > kMaxDv || p.conv_width > kMaxTaps || p.group > 8) return LSC_ERR_UNSUPPORTED;
  const bool bf = ssm_dtype == LSC_BF16;
  switch (dk) {
    case 16: return bf ? dispatch_decode_passes<16, __nv_bfloat16>(p, s) : dispatch_decode_passes<16, float>(p, s);
    case 32: return bf ? dispatch_decode_passes<32, __nv_bfloat16>(p, s) : dispatch_decode_passes<32, float>(p, s);
    case 64: return bf ? dispatch_decode_passes<64, __nv_bfloat16>(p, s) : dispatch_decode_passes<64, float>(p, s);
    case 128: return bf ? dispatch_decode_passes<128, __nv_bfloat16>(p, s) : dispatch_decode_passes<128, float>(p, s);
    default: return LSC_ERR_UNSUPPORTED;
  }
}

int launch_recurrent(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (p.dv > kMaxDv) return LSC_ERR_UNSUPPORTED;
  const bool bf = ssm_dtype == LSC_BF16;
  switch (dk) {
    case 16: return bf ? launch_recurrent_t<16, __nv_bfloat16>(p, s) : launch_recurrent_t<16, float>(p, s);
    case 32: return bf ? launch_recurrent_t<32, __nv_bfloat16>(p, s) : launch_recurrent_t<32, float>(p, s);
    case 64: return bf ? launch_recurrent_t<64, __nv_bfloat16>(p, s) : launch_recurrent_t<64, float>(p, s);
    case 128: return bf ? launch_recurrent_t<128, __nv_bfloat16>(p, s) : launch_recurrent_t<128, float>(p, s);
    default: return LSC_ERR_UNSUPPORTED;
  }
}

}  // namespace lsc
