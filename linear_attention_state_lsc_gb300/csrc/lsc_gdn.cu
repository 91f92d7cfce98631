// lsc_gdn.cu -- the token-by-token GDN recurrence of a resumed prefill, and the
// dispatch of the decode instantiations (lsc_decode_f32.cu, lsc_decode_bf16.cu).
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with
//        q); "相同前缀不一定能全部复用" (continue from the restored checkpoint)
//
// Per token the state update is the delta rule S' = a S (I - b k k^T) + b v k^T
// applied row by row (u_r = S_r.k, d_r = b (v_r - a u_r), S'_r = a S_r + d_r k),
// with o_t = S' q_t.
#include "lsc_gdn_common.cuh"

namespace lsc {

int launch_decode_f32(const DecodeParams &p, int dk, cudaStream_t s);
int launch_decode_bf16(const DecodeParams &p, int dk, cudaStream_t s);

namespace {

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
  return ssm_dtype == LSC_BF16 ? launch_decode_bf16(p, dk, s) : launch_decode_f32(p, dk, s);
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
