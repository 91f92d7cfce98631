// lsc_chunked.cu -- the resumed-prefill GDN recurrence evaluated a chunk of
// tokens at a time: the same token-ordered result as the token-by-token kernel
// (S' = a S (I - b k k^T) + b v k^T, o = S' q per token), rearranged so that
// most of the arithmetic is independent products instead of one dependent
// chain per token.  fp32 on the CUDA cores.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule, the token recurrence)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with
//        q); "相同前缀不一定能全部复用" (continue from the restored checkpoint)
// The pages give the token recurrence only; the chunked form below is its
// algebraic rearrangement, exact up to rounding.
//
// One chunk, tokens 0..C-1, starting from a state row s (length dk):
//   Gam(j,t) = a_(j+1) ... a_t  (Gam(t,t) = 1),   E_t = a_0 ... a_t
//   s after token t = E_t s + sum_{j<=t} Gam(j,t) d_j k_j
// Token t's prediction then needs only s.k_t and the chunk's Gram products:
//   P_t = s.k_t,  R_t = s.q_t,  G_jt = k_j.k_t,  M_jt = k_j.q_t
//   (I + A) d = x,  A_tj = b_t Gam(j,t) G_jt (j < t),  x_t = b_t (v_t - E_t P_t)
//   o_t = E_t R_t + sum_{j<=t} Gam(j,t) M_jt d_j
//   s'  = E_(C-1) s + sum_j Gam(j,C-1) d_j k_j
// A and the Gam-weighted M are the same for every row of the head, so
// T = (I + A)^-1 (unit lower triangular) is formed once per chunk by forward
// substitution, and each row needs P, R (2 C dk products), d = T x, o, and the
// rank-C update (C dk products): about the token kernel's 3 dk products per
// row and token, plus C per row and token for T x and o.
//
// CTA = one (sequence, v head), 256 threads, two CTAs per SM.  The state lives
// in registers as in the token kernel (thread = two rows x 32 columns, four
// threads per row, float pairs for fma.rn.f32x2).  Per chunk:
//   1  the chunk's q, k, v, alpha, beta are in shared memory (cp.async, the
//      next chunk's copies are issued here); tokens past the sequence are
//      padded with k = q = v = 0, alpha = 1, beta = 0, which adds nothing
//   2  each thread forms one Gram entry (120 G_jt, j < t, and 136 M_jt, j <= t)
//      with its Gam factor; every thread forms P and R for its two rows; warp
//      7 forms E_t and Gam(t, C-1)
//   3  warp 0 forms T; every thread forms x for its row's tokens
//   4  thread (row r, parity): d_t = (T x)_t and o_t for its eight tokens of
//      one parity; d_t is scaled by Gam(t, C-1) for the update
//   5  every thread applies s' = E_(C-1) s + sum_t d_t k_t to its two rows
#include "lsc_gdn_common.cuh"

namespace lsc {
namespace {

constexpr int kC = 16;        // tokens per chunk
constexpr int kThreads = 256;
constexpr int kDK = 128;      // head_k_dim of this kernel
constexpr int kKP = kDK + 4;  // row stride (floats) of the q and k tiles: eight rows fall on distinct banks
constexpr int kCP = kC + 4;   // row stride (floats) of the [row][token] and [token][token] arrays
constexpr int kRows = kMaxDv; // rows of the per-row arrays

__host__ __device__ inline int chunk_buf_floats(int dv) {
  // q [C][KP], k [C][KP], v [C][dv], alpha [C], beta [C]; a multiple of 4 floats
  return (2 * kC * kKP + kC * dv + 2 * kC + 3) / 4 * 4;
}
constexpr int kArrFloats = 3 * kRows * kCP + 2 * kC * kCP + kC * kCP + 2 * kC;
__host__ __device__ inline int64_t chunk_smem_bytes(int dv) {
  return (2 * (int64_t)chunk_buf_floats(dv) + kArrFloats) * 4;
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

template <typename TS>
__global__ void __launch_bounds__(kThreads, 2) recurrent_chunked_kernel(const __grid_constant__ RecurrentParams p) {
  extern __shared__ __align__(16) float csm[];
  __shared__ int32_t s_len[kRankedSeqs];
  __shared__ int32_t s_seq;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, g = h / p.group;
  const int dv = p.dv;
  const int buf = chunk_buf_floats(dv);
  float *const arr = csm + 2 * buf;
  float *const P_s = arr;                    // [row][t]: P_t, then x_t in place
  float *const R_s = P_s + kRows * kCP;      // [row][t]: R_t
  float *const D_s = R_s + kRows * kCP;      // [row][t]: d_t, then Gam(t, C-1) d_t
  float *const At_s = D_s + kRows * kCP;     // [j][t]: A_tj (j < t), transposed
  float *const B_s = At_s + kC * kCP;        // [t][j]: Gam(j,t) M_jt (j <= t)
  float *const T_s = B_s + kC * kCP;         // [t][j]: (I + A)^-1
  float *const E_s = T_s + kC * kCP;         // [t]: a_0 ... a_t
  float *const F_s = E_s + kC;               // [t]: Gam(t, C-1)

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
    for (int64_t e = tid; e < (int64_t)(t1 - t0) * dv; e += kThreads) {
      const int64_t t = t0 + e / dv;
      p.out[(t * p.Hv + h) * dv + e % dv] = 0.f;
    }
    return;
  }

  // The upper triangles of A and B and the rows >= dv of P, R, D are never
  // written: they stay zero.
  for (int e = tid; e < kArrFloats; e += kThreads) arr[e] = 0.f;

  // state layout: rows rp and rp + rh, float4 columns lr, lr + 4, ... of each
  const int lr = tid & 3, rp = tid >> 2;
  const int rh = (dv + 1) / 2;
  const int rows[2] = {rp, rp + rh};
  bool rv[2];
  rv[0] = rp < rh && rows[0] < dv;
  rv[1] = rp < rh && rows[1] < dv;
  uint64_t S[2][16];
  TS *Sg = reinterpret_cast<TS *>(p.layer + (int64_t)slot * p.page + p.ssm_off) + (int64_t)h * dv * kDK;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
#pragma unroll
    for (int jv = 0; jv < 8; ++jv) {
      const int c0 = (jv * 4 + lr) * 4;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = 0.f;
        if (warm && rv[q]) {
          if constexpr (sizeof(TS) == 4) v[e] = ((const float *)Sg)[(int64_t)rows[q] * kDK + c0 + e];
          else v[e] = bf16_bits_to_float(((const uint16_t *)Sg)[(int64_t)rows[q] * kDK + c0 + e]);
        }
      }
      S[q][jv * 2] = f2_pack(v[0], v[1]);
      S[q][jv * 2 + 1] = f2_pack(v[2], v[3]);
    }
  }
  // solve layout: row r, tokens of parity pr
  const int r = tid >> 1, pr = tid & 1;

  const bool v16 = (dv % 4 == 0) && (((uintptr_t)p.v & 15) == 0);
  auto issue_tile = [&](int tb, int bsel) {
    const int nt = min(kC, t1 - tb);
    float *qd = csm + bsel * buf, *kd = qd + kC * kKP, *vd = kd + kC * kKP;
    float *ad = vd + kC * dv, *bd = ad + kC;
    for (int e = tid; e < nt * (kDK / 4); e += kThreads) {
      const int tt = e / (kDK / 4), c4 = e % (kDK / 4);
      const int64_t src = ((int64_t)(tb + tt) * p.Hk + g) * kDK + c4 * 4;
      cp_async16(qd + tt * kKP + c4 * 4, p.q + src);
      cp_async16(kd + tt * kKP + c4 * 4, p.k + src);
    }
    if (v16) {
      for (int e = tid; e < nt * (dv / 4); e += kThreads) {
        const int tt = e / (dv / 4), c4 = e % (dv / 4);
        cp_async16(vd + tt * dv + c4 * 4, p.v + ((int64_t)(tb + tt) * p.Hv + h) * dv + c4 * 4);
      }
    } else {
      for (int e = tid; e < nt * dv; e += kThreads) {
        const int tt = e / dv, c = e % dv;
        cp_async4(vd + tt * dv + c, p.v + ((int64_t)(tb + tt) * p.Hv + h) * dv + c);
      }
    }
    if (tid < nt) {
      cp_async4(ad + tid, p.alpha + (int64_t)(tb + tid) * p.Hv + h);
      cp_async4(bd + tid, p.beta + (int64_t)(tb + tid) * p.Hv + h);
    }
  };

  if (t0 < t1) issue_tile(t0, 0);
  cp_async_commit();
  int bsel = 0;
  for (int cb = t0; cb < t1; cb += kC, bsel ^= 1) {
    const int nt = min(kC, t1 - cb);
    float *const qd = csm + bsel * buf, *const kd = qd + kC * kKP, *const vd = kd + kC * kKP;
    float *const ad = vd + kC * dv, *const bd = ad + kC;
    cp_async_wait<0>();
    if (nt < kC) {  // tokens past the sequence: k = q = v = 0, alpha = 1, beta = 0
      for (int e = tid; e < (kC - nt) * kKP; e += kThreads) {
        qd[nt * kKP + e] = 0.f;
        kd[nt * kKP + e] = 0.f;
      }
      for (int e = tid; e < (kC - nt) * dv; e += kThreads) vd[nt * dv + e] = 0.f;
      if (tid < kC - nt) {
        ad[nt + tid] = 1.f;
        bd[nt + tid] = 0.f;
      }
    }
    __syncthreads();  // (1) the chunk is in shared memory; every thread is done with the previous one
    if (cb + kC < t1) issue_tile(cb + kC, bsel ^ 1);
    cp_async_commit();

    // (2a) E_t and Gam(t, C-1)
    if (warp == 7 && lane < kC) {
      float e = 1.f, f = 1.f;
#pragma unroll
      for (int t = 0; t < kC; ++t) {
        if (t <= lane) e *= ad[t];
        if (t > lane) f *= ad[t];
      }
      E_s[lane] = e;
      F_s[lane] = f;
    }
    // (2b) one Gram entry per thread, with its Gam factor: tid < 120 -> G_jt
    // (j < t) as A_tj; else M_jt (j <= t) as B_tj
    {
      constexpr int nG = kC * (kC - 1) / 2;
      const bool isG = tid < nG;
      const int e = isG ? tid : tid - nG;
      int t = isG ? 1 : 0;  // row t starts at t(t-1)/2 (G) or t(t+1)/2 (M)
      while (t + 1 < kC && (isG ? (t + 1) * t / 2 : (t + 1) * (t + 2) / 2) <= e) ++t;
      const int j = e - (isG ? t * (t - 1) / 2 : t * (t + 1) / 2);
      const float *a = kd + j * kKP, *b = (isG ? kd : qd) + t * kKP;
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll 8
      for (int c = 0; c < kDK; c += 8) {
        const ulonglong2 x0 = *reinterpret_cast<const ulonglong2 *>(a + c);
        const ulonglong2 y0 = *reinterpret_cast<const ulonglong2 *>(b + c);
        const ulonglong2 x1 = *reinterpret_cast<const ulonglong2 *>(a + c + 4);
        const ulonglong2 y1 = *reinterpret_cast<const ulonglong2 *>(b + c + 4);
        acc0 = f2_fma(x0.x, y0.x, acc0);
        acc1 = f2_fma(x0.y, y0.y, acc1);
        acc0 = f2_fma(x1.x, y1.x, acc0);
        acc1 = f2_fma(x1.y, y1.y, acc1);
      }
      float l0, h0, l1, h1;
      f2_unpack(acc0, l0, h0);
      f2_unpack(acc1, l1, h1);
      float gm = 1.f;  // Gam(j, t)
      for (int m = j + 1; m <= t; ++m) gm *= ad[m];
      const float dot = (l0 + h0) + (l1 + h1);
      if (isG) At_s[j * kCP + t] = bd[t] * gm * dot;
      else B_s[t * kCP + j] = gm * dot;
    }
    // (2c) P_t = s.k_t and R_t = s.q_t for the thread's two rows, two tokens at
    // a time; the four partial sums of a row are reduced so that lane lr ends
    // with (kind lr >> 1, row lr & 1) of both tokens
#pragma unroll 1
    for (int ta = 0; ta < kC; ta += 2) {
      uint64_t acc[8];  // [kind][row][token]
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0;
#pragma unroll
      for (int jv = 0; jv < 8; ++jv) {
        const int c0 = (jv * 4 + lr) * 4;
        const ulonglong2 ka = *reinterpret_cast<const ulonglong2 *>(kd + ta * kKP + c0);
        const ulonglong2 kb = *reinterpret_cast<const ulonglong2 *>(kd + (ta + 1) * kKP + c0);
        const ulonglong2 qa = *reinterpret_cast<const ulonglong2 *>(qd + ta * kKP + c0);
        const ulonglong2 qb = *reinterpret_cast<const ulonglong2 *>(qd + (ta + 1) * kKP + c0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint64_t s0 = S[q][jv * 2], s1 = S[q][jv * 2 + 1];
          acc[q * 2] = f2_fma(s1, ka.y, f2_fma(s0, ka.x, acc[q * 2]));
          acc[q * 2 + 1] = f2_fma(s1, kb.y, f2_fma(s0, kb.x, acc[q * 2 + 1]));
          acc[4 + q * 2] = f2_fma(s1, qa.y, f2_fma(s0, qa.x, acc[4 + q * 2]));
          acc[4 + q * 2 + 1] = f2_fma(s1, qb.y, f2_fma(s0, qb.x, acc[4 + q * 2 + 1]));
        }
      }
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float lo, hi;
        f2_unpack(acc[e], lo, hi);
        v[e] = lo + hi;
      }
      const bool b1 = (lr >> 1) != 0, b0 = (lr & 1) != 0;
      float k4[4];  // kind b1: [row][token]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float send = b1 ? v[e] : v[4 + e];
        const float keep = b1 ? v[4 + e] : v[e];
        k4[e] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      float k2[2];  // kind b1, row b0: [token]
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float send = b0 ? k4[e] : k4[2 + e];
        const float keep = b0 ? k4[2 + e] : k4[e];
        k2[e] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
      const int row = b0 ? rows[1] : rows[0];
      if (b0 ? rv[1] : rv[0])
        *reinterpret_cast<float2 *>((b1 ? R_s : P_s) + row * kCP + ta) = make_float2(k2[0], k2[1]);
    }
    __syncthreads();  // (2)

    // (3a) x_t = b_t (v_t - E_t P_t) for row r, tokens of parity pr (in place of P)
    if (r < dv) {
#pragma unroll
      for (int u = 0; u < kC / 2; ++u) {
        const int t = 2 * u + pr;
        P_s[r * kCP + t] = bd[t] * (vd[t * dv + r] - E_s[t] * P_s[r * kCP + t]);
      }
    }
    // (3b) T = (I + A)^-1, one column per lane: T_mj = [m == j] - sum_{j<=n<m} A_mn T_nj,
    // each finished entry is folded into the sums of the later rows
    if (warp == 0 && lane < kC) {
      const int j = lane;
      float acc[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t) acc[t] = 0.f;
#pragma unroll
      for (int m = 0; m < kC; ++m) {
        const float tm = m == j ? 1.f : (m > j ? -acc[m] : 0.f);
        T_s[m * kCP + j] = tm;
#pragma unroll
        for (int t4 = (m + 1) / 4 * 4; t4 < kC; t4 += 4) {
          const float4 a4 = *reinterpret_cast<const float4 *>(At_s + m * kCP + t4);
          const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (t4 + e > m) acc[t4 + e] = fmaf(av[e], tm, acc[t4 + e]);
        }
      }
    }
    const float e_last = E_s[kC - 1];
    __syncthreads();  // (3)

    // (4) d = T x and o for row r, tokens of parity pr; then d_t *= Gam(t, C-1)
    {
      const float4 *xr = reinterpret_cast<const float4 *>(P_s + r * kCP);
      const float4 *dr = reinterpret_cast<const float4 *>(D_s + r * kCP);
#pragma unroll
      for (int u = 0; u < kC / 2; ++u) {
        const int t = 2 * u + pr;
        const float4 *tr = reinterpret_cast<const float4 *>(T_s + t * kCP);
        float d = 0.f;
#pragma unroll
        for (int w4 = 0; w4 <= u / 2; ++w4) d = dot4(tr[w4], xr[w4], d);  // T_tj = 0 for j > t
        D_s[r * kCP + t] = d;
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < kC / 2; ++u) {
        const int t = 2 * u + pr;
        const float4 *br = reinterpret_cast<const float4 *>(B_s + t * kCP);
        float o = E_s[t] * R_s[r * kCP + t];
#pragma unroll
        for (int w4 = 0; w4 <= u / 2; ++w4) o = dot4(br[w4], dr[w4], o);  // B_tj = 0 for j > t
        if (t < nt && r < dv) p.out[((int64_t)(cb + t) * p.Hv + h) * dv + r] = o;
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < kC / 2; ++u) {
        const int t = 2 * u + pr;
        D_s[r * kCP + t] *= F_s[t];
      }
    }
    __syncthreads();  // (4)

    // (5) s' = E_(C-1) s + sum_t d_t k_t
    {
      const uint64_t el = f2_pack(e_last, e_last);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int c = 0; c < 16; ++c) S[q][c] = f2_mul(S[q][c], el);
#pragma unroll 1
      for (int t4 = 0; t4 < kC; t4 += 4) {
        const float4 da = *reinterpret_cast<const float4 *>(D_s + rows[0] * kCP + t4);
        const float4 db = *reinterpret_cast<const float4 *>(D_s + rows[1] * kCP + t4);
        const float dva[4] = {da.x, da.y, da.z, da.w}, dvb[4] = {db.x, db.y, db.z, db.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint64_t d0 = f2_pack(dva[e], dva[e]), d1 = f2_pack(dvb[e], dvb[e]);
          const float *kt = kd + (t4 + e) * kKP;
#pragma unroll
          for (int jv = 0; jv < 8; ++jv) {
            const ulonglong2 k4 = *reinterpret_cast<const ulonglong2 *>(kt + (jv * 4 + lr) * 4);
            S[0][jv * 2] = f2_fma(d0, k4.x, S[0][jv * 2]);
            S[0][jv * 2 + 1] = f2_fma(d0, k4.y, S[0][jv * 2 + 1]);
            S[1][jv * 2] = f2_fma(d1, k4.x, S[1][jv * 2]);
            S[1][jv * 2 + 1] = f2_fma(d1, k4.y, S[1][jv * 2 + 1]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int q = 0; q < 2; ++q) {
    if (!rv[q]) continue;
#pragma unroll
    for (int jv = 0; jv < 8; ++jv) {
      const int c0 = (jv * 4 + lr) * 4;
      float f[4];
      f2_unpack(S[q][jv * 2], f[0], f[1]);
      f2_unpack(S[q][jv * 2 + 1], f[2], f[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (sizeof(TS) == 4) ((float *)Sg)[(int64_t)rows[q] * kDK + c0 + e] = f[e];
        else ((uint16_t *)Sg)[(int64_t)rows[q] * kDK + c0 + e] = float_to_bf16_bits(f[e]);
      }
    }
  }
}

template <typename TS>
int launch_chunked_t(const RecurrentParams &p, cudaStream_t s) {
  const int64_t smem = chunk_smem_bytes(p.dv);
  static SmemLimit limit;  // per instantiation and device
  if (limit.ensure((const void *)recurrent_chunked_kernel<TS>, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  recurrent_chunked_kernel<TS><<<dim3(p.Hv, p.n_seq, 1), kThreads, (size_t)smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace

int launch_recurrent_chunked(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (dk != kDK || p.dv > kMaxDv || p.dv < 1) return LSC_ERR_UNSUPPORTED;
  return ssm_dtype == LSC_BF16 ? launch_chunked_t<__nv_bfloat16>(p, s) : launch_chunked_t<float>(p, s);
}

}  // namespace lsc
