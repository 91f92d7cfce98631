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
// Token-by-token recurrence for head_k_dim 16, 32 and 64 (128 has its own
// kernel with eight rows per thread, lsc_rec128.cu).  Grid (Hv, n_seq), one
// CTA per (sequence, v head), 2 CTAs per SM.  Each thread keeps two rows of
// the head's state (CPT columns of each, TPR threads per row) in registers for
// the whole sequence.
//
// The state is held scaled, S = gamma * Shat, so that a token costs three
// FMAs per element: Shat.k and Shat.q for the row's prediction and read-out,
// then Shat += (d / gamma') k with gamma' = alpha * gamma.  Per row
//   u = gamma (Shat.k),  d = beta (v - alpha u),  o = gamma' (Shat.q) + d (k.q),
// which is S' = alpha S + d k^T and o = S' q.  When gamma' falls below 2^-32
// (or alpha is 0) the scale is folded into Shat and gamma restarts at 1; at the
// end the state is stored as gamma * Shat.
// Tokens are staged TT at a time with cp.async, double-buffered, and k.q of
// each token is formed once per tile.  When there are at most kRankedSeqs
// sequences, CTAs take them longest first so that long sequences do not finish
// last.
constexpr int kTileTokens = 32;
constexpr int kRecThreads = 256;

template <int DK>
struct RecShape {
  static constexpr int CPT = DK < 32 ? DK : 32;  // columns per thread
  static constexpr int TPR = DK / CPT;           // threads per row
  static constexpr int NV4 = CPT / 4;            // float4 vectors per thread per row
};

__host__ __device__ inline int64_t rec_smem_bytes(int dk, int dv) {
  // two buffers of: q, k [TT][dk], v [TT][dv], alpha, beta, k.q [TT]
  return 2 * ((int64_t)kTileTokens * (2 * dk + dv) + 3 * kTileTokens) * 4;
}

template <int DK, typename TS>
__global__ void __launch_bounds__(kRecThreads, 2) recurrent_kernel(const __grid_constant__ RecurrentParams p) {
  using R = RecShape<DK>;
  constexpr int TT = kTileTokens;
  extern __shared__ __align__(16) float rsm[];
  __shared__ int32_t s_len[kRankedSeqs];
  __shared__ int32_t s_seq;

  const int tid = threadIdx.x;
  const int h = blockIdx.x, g = h / p.group;
  const int dv = p.dv;
  const int buf_floats = TT * (2 * DK + dv) + 3 * TT;
  auto q_s = [&](int b) { return rsm + b * buf_floats; };
  auto k_s = [&](int b) { return rsm + b * buf_floats + TT * DK; };
  auto v_s = [&](int b) { return rsm + b * buf_floats + 2 * TT * DK; };
  auto a_s = [&](int b) { return rsm + b * buf_floats + TT * (2 * DK + dv); };
  auto b_s = [&](int b) { return a_s(b) + TT; };
  auto kq_s = [&](int b) { return a_s(b) + 2 * TT; };

  const int i = ranked_sequence(p.cu, p.n_seq, s_len, &s_seq);

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
  if (!valid) {  // uniform over the CTA
    for (int64_t e = tid; e < (int64_t)(t1 - t0) * dv; e += kRecThreads) {
      const int64_t t = t0 + e / dv;
      p.out[(t * p.Hv + h) * dv + e % dv] = 0.f;
    }
    return;
  }

  const int lr = tid % R::TPR;
  const int rp = tid / R::TPR;     // row pair
  const int rh = (dv + 1) / 2;     // rows rp and rp + rh
  const int rows[2] = {rp, rp + rh};
  bool rv[2];
  rv[0] = rp < rh && rows[0] < dv;
  rv[1] = rp < rh && rows[1] < dv;

  // state rows into registers, as float pairs for the f32x2 arithmetic
  constexpr int NP = R::CPT / 2;
  uint64_t S[2][NP];
  TS *Sg = reinterpret_cast<TS *>(p.layer + (int64_t)slot * p.page + p.ssm_off) + (int64_t)h * dv * DK;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int jv = 0; jv < R::NV4; ++jv) {
      const int c0 = (jv * R::TPR + lr) * 4;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = 0.f;
        if (warm && rv[q]) {
          if constexpr (sizeof(TS) == 4) v[e] = ((const float *)Sg)[(int64_t)rows[q] * DK + c0 + e];
          else v[e] = bf16_bits_to_float(((const uint16_t *)Sg)[(int64_t)rows[q] * DK + c0 + e]);
        }
      }
      S[q][jv * 2] = f2_pack(v[0], v[1]);
      S[q][jv * 2 + 1] = f2_pack(v[2], v[3]);
    }
  }
  float gam = 1.f;

  const bool v16 = (dv % 4 == 0) && (((uintptr_t)p.v & 15) == 0);
  auto issue_tile = [&](int tb, int bsel) {
    const int nt = min(TT, t1 - tb);
    float *qd = q_s(bsel), *kd = k_s(bsel), *vd = v_s(bsel);
    for (int e = tid; e < nt * (DK / 4); e += kRecThreads) {
      const int tt = e / (DK / 4), c4 = e % (DK / 4);
      const int64_t src = ((int64_t)(tb + tt) * p.Hk + g) * DK + c4 * 4;
      cp_async16(qd + tt * DK + c4 * 4, p.q + src);
      cp_async16(kd + tt * DK + c4 * 4, p.k + src);
    }
    if (v16) {
      for (int e = tid; e < nt * (dv / 4); e += kRecThreads) {
        const int tt = e / (dv / 4), c4 = e % (dv / 4);
        cp_async16(vd + tt * dv + c4 * 4, p.v + ((int64_t)(tb + tt) * p.Hv + h) * dv + c4 * 4);
      }
    } else {
      for (int e = tid; e < nt * dv; e += kRecThreads) {
        const int tt = e / dv, c = e % dv;
        cp_async4(vd + tt * dv + c, p.v + ((int64_t)(tb + tt) * p.Hv + h) * dv + c);
      }
    }
    if (tid < nt) {
      cp_async4(a_s(bsel) + tid, p.alpha + (int64_t)(tb + tid) * p.Hv + h);
      cp_async4(b_s(bsel) + tid, p.beta + (int64_t)(tb + tid) * p.Hv + h);
    }
  };

  if (t0 < t1) issue_tile(t0, 0);
  cp_async_commit();
  const int warp = tid >> 5, lane = tid & 31;
  int bsel = 0;
  for (int tb = t0; tb < t1; tb += TT, bsel ^= 1) {
    const int nt = min(TT, t1 - tb);
    if (tb + TT < t1) issue_tile(tb + TT, bsel ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of the current tile have landed
    __syncthreads();
    const float *qd = q_s(bsel), *kd = k_s(bsel), *vd = v_s(bsel);
    for (int tt = warp; tt < nt; tt += kRecThreads / 32) {
      float acc = 0.f;
      for (int c = lane; c < DK; c += 32) acc = fmaf(qd[tt * DK + c], kd[tt * DK + c], acc);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      if (lane == 0) kq_s(bsel)[tt] = acc;
    }
    __syncthreads();
    const float *al = a_s(bsel), *be = b_s(bsel), *kq = kq_s(bsel);
    for (int tt = 0; tt < nt; ++tt) {
      const float *kt = kd + tt * DK, *qt = qd + tt * DK;
      uint64_t kr[NP];
      uint64_t u2[2] = {0, 0}, w2[2] = {0, 0};  // (even, odd) column partial sums
#pragma unroll
      for (int jv = 0; jv < R::NV4; ++jv) {
        const int c0 = (jv * R::TPR + lr) * 4;
        const ulonglong2 k4 = *reinterpret_cast<const ulonglong2 *>(kt + c0);
        const ulonglong2 q4 = *reinterpret_cast<const ulonglong2 *>(qt + c0);
        kr[jv * 2] = k4.x;
        kr[jv * 2 + 1] = k4.y;
        const uint64_t qa = q4.x, qb = q4.y;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          u2[q] = f2_fma(S[q][jv * 2], kr[jv * 2], u2[q]);
          u2[q] = f2_fma(S[q][jv * 2 + 1], kr[jv * 2 + 1], u2[q]);
          w2[q] = f2_fma(S[q][jv * 2], qa, w2[q]);
          w2[q] = f2_fma(S[q][jv * 2 + 1], qb, w2[q]);
        }
      }
      float u[2], w[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float lo, hi;
        f2_unpack(u2[q], lo, hi);
        u[q] = lo + hi;
        f2_unpack(w2[q], lo, hi);
        w[q] = lo + hi;
      }
#pragma unroll
      for (int m = R::TPR / 2; m >= 1; m >>= 1) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          u[q] += __shfl_xor_sync(0xffffffffu, u[q], m);
          w[q] += __shfl_xor_sync(0xffffffffu, w[q], m);
        }
      }
      const float a = al[tt], b = be[tt];
      float gn = a * gam;  // gamma' = alpha gamma
      float d[2], o[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float vr = rv[q] ? vd[tt * dv + rows[q]] : 0.f;
        d[q] = b * (vr - a * (gam * u[q]));
        o[q] = fmaf(gn, w[q], d[q] * kq[tt]);
      }
      if (gn < 0x1p-32f) {  // fold the scale into Shat (uniform over the CTA)
        const uint64_t g2 = f2_pack(gn, gn);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int c = 0; c < NP; ++c) S[q][c] = f2_mul(S[q][c], g2);
        gn = 1.f;
      }
      const float inv = 1.f / gn;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float e = d[q] * inv;
        const uint64_t e2 = f2_pack(e, e);
#pragma unroll
        for (int c = 0; c < NP; ++c) S[q][c] = f2_fma(e2, kr[c], S[q][c]);
      }
      gam = gn;
      if (lr == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (rv[q]) p.out[((int64_t)(tb + tt) * p.Hv + h) * dv + rows[q]] = o[q];
      }
    }
    __syncthreads();  // the next iteration refills this buffer
  }
  cp_async_wait<0>();

  // final state = gamma * Shat
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    if (!rv[q]) continue;
#pragma unroll
    for (int jv = 0; jv < R::NV4; ++jv) {
      const int c0 = (jv * R::TPR + lr) * 4;
      float f[4];
      f2_unpack(S[q][jv * 2], f[0], f[1]);
      f2_unpack(S[q][jv * 2 + 1], f[2], f[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = gam * f[e];
        if constexpr (sizeof(TS) == 4) ((float *)Sg)[(int64_t)rows[q] * DK + c0 + e] = v;
        else ((uint16_t *)Sg)[(int64_t)rows[q] * DK + c0 + e] = float_to_bf16_bits(v);
      }
    }
  }
}

template <int DK, typename TS>
int launch_recurrent_t(const RecurrentParams &p, cudaStream_t s) {
  using R = RecShape<DK>;
  if ((p.dv + 1) / 2 * R::TPR > kRecThreads) return LSC_ERR_UNSUPPORTED;
  const int64_t smem = rec_smem_bytes(DK, p.dv);
  static SmemLimit limit;  // per instantiation and device
  if (limit.ensure((const void *)recurrent_kernel<DK, TS>, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  recurrent_kernel<DK, TS><<<dim3(p.Hv, p.n_seq, 1), kRecThreads, (size_t)smem, s>>>(p);
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
    case 128: return launch_recurrent128(p, ssm_dtype, s);  // eight rows per thread (lsc_rec128.cu)
    default: return LSC_ERR_UNSUPPORTED;
  }
}

}  // namespace lsc
