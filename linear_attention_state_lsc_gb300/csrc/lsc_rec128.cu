// lsc_rec128.cu -- the token-by-token GDN recurrence of a resumed prefill for
// head_k_dim 128, with eight state rows per thread.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with
//        q); "相同前缀不一定能全部复用" (continue from the restored checkpoint)
//
// Per token and state row r: u = S_r.k, d = b (v_r - a u), S_r <- a S_r + d k,
// o_r = S_r.q (after the update), with the state held scaled (S = gamma Shat)
// as in the general token kernel of lsc_gdn.cu: u = gamma (Shat.k),
// o = gamma' (Shat.q) + d (k.q), Shat += (d / gamma') k, gamma' = a gamma.
//
// Why a second token kernel: every token's k and q must reach every thread
// that holds state, through shared memory, and a 128-bit shared load costs
// four wavefronts whether or not its lanes share addresses.  With two rows x
// 32 columns per thread each loaded k or q value feeds two rows, and shared
// memory (not the FP32 pipe) sets the pace.  Here a thread holds 8 rows x 8
// columns (its 16-lane group covers 8 full rows): each loaded value feeds
// eight rows, four times fewer wavefronts per flop.  The price is a 16-lane
// reduction per token: the 16 dot products of the thread (u and w of 8 rows)
// are reduce-scattered in four shuffle rounds so that lane l of the group ends
// with value l (u of row l/2 on even lanes, w on odd lanes), and the eight d
// values are then broadcast back with indexed shuffles.  Each lane keeps its
// values in the order (value index) XOR (its lane index): row r of the group
// sits in register slot r ^ (l >> 1) and odd lanes form the q products first,
// so every round keeps the lower half and sends the upper one, with no
// lane-dependent selects.
//
// Tokens go in pairs (a, b): both tokens' dot products are formed against the
// state before the pair (one token after the other, so that the 64 state
// registers, one token's inputs and its 16 products fit in 128 registers with
// nothing spilled), and b's are corrected with the pair's Gram scalars (true
// state S = gamma Shat; gamma_a' = alpha_a gamma, gamma_b' = alpha_b gamma_a'):
//   d_a = beta_a (v_a - gamma_a' Shat.k_a),  o_a = gamma_a' Shat.q_a + d_a (k_a.q_a)
//   u_b = gamma_a' Shat.k_b + d_a (k_a.k_b), d_b = beta_b (v_b - alpha_b u_b)
//   o_b = gamma_b' Shat.q_b + alpha_b d_a (k_a.q_b) + d_b (k_b.q_b)
//   Shat += (d_a / gamma_a') k_a + (d_b / gamma_b') k_b
// which is the token recurrence applied twice.  When gamma_a' or gamma_b'
// falls below 2^-32 the pair folds the scale into the state instead:
// Shat = gamma_b' Shat + alpha_b d_a k_a + d_b k_b, gamma = 1 (no division).
// An odd tile ends with a pair whose second token is empty (k = q = v = 0,
// alpha = 1, beta = 0).  The pair scalars depend on alpha alone and are
// formed once per tile; k.q, k_a.k_b and k_a.q_b by the other warps.
//
// CTA = one (sequence, v head), 256 threads = 16 groups, two CTAs per SM;
// tokens staged 32 at a time with cp.async, double-buffered, k.q formed once
// per token; with at most 256 sequences the CTAs take them longest first.
#include "lsc_gdn_common.cuh"

namespace lsc {
namespace {

constexpr int kTT = 32;  // tokens per tile
constexpr int kThreads = 256;
constexpr int kDK = 128;

__host__ __device__ inline int rec128_buf_floats(int dv) {
  // one buffer: q, k [TT][dk], per-pair scalars float4 [TT] (two per pair),
  // v [TT][dv], alpha, beta, k.q [TT], per-pair Gram scalars [TT] (two per pair)
  return kTT * (2 * kDK + 4 + dv) + 4 * kTT;
}
__host__ __device__ inline int64_t rec128_smem_bytes(int dv) { return 2 * (int64_t)rec128_buf_floats(dv) * 4; }

// Two float pairs as the sum of their four floats' products: a.b over 4 columns.
__device__ __forceinline__ float dot8(const uint64_t *s, const uint64_t *x) {
  uint64_t acc = f2_mul(s[0], x[0]);
  acc = f2_fma(s[1], x[1], acc);
  acc = f2_fma(s[2], x[2], acc);
  acc = f2_fma(s[3], x[3], acc);
  float lo, hi;
  f2_unpack(acc, lo, hi);
  return lo + hi;
}

// One round of the reduce-scatter over lanes l and l ^ m, in the lane-permuted
// order: keep the lower half, add the partner's upper half.
template <int N>
__device__ __forceinline__ void reduce_half(const float *v, float *out, int m) {
#pragma unroll
  for (int e = 0; e < N / 2; ++e) out[e] = v[e] + __shfl_xor_sync(0xffffffffu, v[N / 2 + e], m);
}

template <typename TS>
__global__ void __launch_bounds__(kThreads, 2) recurrent128_kernel(const __grid_constant__ RecurrentParams p) {
  extern __shared__ __align__(16) float rsm[];
  __shared__ int32_t s_len[kRankedSeqs];
  __shared__ int32_t s_seq;
  __shared__ float s_gam;

  const int tid = threadIdx.x;
  const int h = blockIdx.x, g = h / p.group;
  const int dv = p.dv;
  const int buf_floats = rec128_buf_floats(dv);
  auto q_s = [&](int b) { return rsm + b * buf_floats; };
  auto k_s = [&](int b) { return rsm + b * buf_floats + kTT * kDK; };
  auto sc_s = [&](int b) { return reinterpret_cast<float4 *>(rsm + b * buf_floats + 2 * kTT * kDK); };
  auto v_s = [&](int b) { return rsm + b * buf_floats + 2 * kTT * kDK + 4 * kTT; };
  auto a_s = [&](int b) { return rsm + b * buf_floats + kTT * (2 * kDK + 4 + dv); };
  auto b_s = [&](int b) { return a_s(b) + kTT; };
  auto kq_s = [&](int b) { return a_s(b) + 2 * kTT; };
  auto gr_s = [&](int b) { return reinterpret_cast<float2 *>(a_s(b) + 3 * kTT); };

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

  // group gr: rows 8 gr .. 8 gr + 7; lane lc: float4 column units lc and lc + 16
  const int lane = tid & 31, lc = tid & 15;
  const int row0 = (tid >> 4) * 8;
  const int rb = lc >> 1;               // register slot r holds row row0 + (r ^ rb)
  const int my_row = row0 + rb;         // after the reduction: u (even lc) or w (odd lc) of this row
  const int gbase = lane & 16;          // the group's first lane in the warp
  const bool odd = (lc & 1) != 0;

  uint64_t S[8][4];  // [slot][pair]: columns 4lc..4lc+3, then 64+4lc..64+4lc+3
  auto state_ptr = [&]() {  // formed where used, so that no register holds it across the token loop
    return reinterpret_cast<TS *>(p.layer + (int64_t)slot * p.page + p.ssm_off) + (int64_t)h * dv * kDK;
  };
  const TS *Sg = state_ptr();
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = row0 + (r ^ rb);
    const bool live = warm && row < dv;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c0 = (lc + 16 * u) * 4;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = 0.f;
        if (live) {
          if constexpr (sizeof(TS) == 4) v[e] = ((const float *)Sg)[(int64_t)row * kDK + c0 + e];
          else v[e] = bf16_bits_to_float(((const uint16_t *)Sg)[(int64_t)row * kDK + c0 + e]);
        }
      }
      S[r][2 * u] = f2_pack(v[0], v[1]);
      S[r][2 * u + 1] = f2_pack(v[2], v[3]);
    }
  }
  float gam = 1.f;

  const bool v16 = (dv % 4 == 0) && (((uintptr_t)p.v & 15) == 0);
  auto issue_tile = [&](int tb, int bsel) {
    const int nt = min(kTT, t1 - tb);
    float *qd = q_s(bsel), *kd = k_s(bsel), *vd = v_s(bsel);
    for (int e = tid; e < nt * (kDK / 4); e += kThreads) {
      const int tt = e / (kDK / 4), c4 = e % (kDK / 4);
      const int64_t src = ((int64_t)(tb + tt) * p.Hk + g) * kDK + c4 * 4;
      cp_async16(qd + tt * kDK + c4 * 4, p.q + src);
      cp_async16(kd + tt * kDK + c4 * 4, p.k + src);
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
      cp_async4(a_s(bsel) + tid, p.alpha + (int64_t)(tb + tid) * p.Hv + h);
      cp_async4(b_s(bsel) + tid, p.beta + (int64_t)(tb + tid) * p.Hv + h);
    }
  };

  if (t0 < t1) issue_tile(t0, 0);
  cp_async_commit();
  const int warp = tid >> 5;
  int bsel = 0;
  for (int tb = t0; tb < t1; tb += kTT, bsel ^= 1) {
    const int nt = min(kTT, t1 - tb);
    if (tb + kTT < t1) issue_tile(tb + kTT, bsel ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // this thread's copies of the current tile have landed
    const int np = (nt + 1) / 2;  // token pairs; an odd tile ends with a pair whose second token is empty
    if (nt & 1) {                 // the empty token: k = q = v = 0, alpha = 1, beta = 0
      for (int e = tid; e < kDK; e += kThreads) {
        q_s(bsel)[nt * kDK + e] = 0.f;
        k_s(bsel)[nt * kDK + e] = 0.f;
      }
      for (int e = tid; e < dv; e += kThreads) v_s(bsel)[nt * dv + e] = 0.f;
      if (tid == 0) {
        a_s(bsel)[nt] = 1.f;
        b_s(bsel)[nt] = 0.f;
      }
    }
    __syncthreads();
    const float *qd = q_s(bsel), *kd = k_s(bsel), *vd = v_s(bsel);
    float4 *sp = sc_s(bsel);
    float2 *gr = gr_s(bsel);
    if (warp == 0) {
      // per pair (tokens a, b): {gamma_a', gamma_b', beta_a, beta_b} and
      // {alpha_b, e-scale of a, e-scale of b, fold}; gamma_a' = alpha_a gamma,
      // gamma_b' = alpha_b gamma_a'.  Below 2^-32 the pair folds the scale into
      // the state (fold = gamma_b', e-scales alpha_b and 1, gamma restarts at 1);
      // otherwise the e-scales are 1 / gamma_a', 1 / gamma_b' and fold is NaN
      if (lane == 0) {
        const float *al = a_s(bsel), *be = b_s(bsel);
        for (int pp = 0; pp < np; ++pp) {
          const float aa = al[2 * pp], ab = al[2 * pp + 1];
          const float ga = aa * gam, gb = ab * ga;
          const bool fold = fminf(ga, gb) < 0x1p-32f;
          sp[2 * pp] = make_float4(ga, gb, be[2 * pp], be[2 * pp + 1]);
          sp[2 * pp + 1] = make_float4(ab, fold ? ab : 0.f, 1.f, fold ? gb : __int_as_float(0x7fffffff));
          gam = fold ? 1.f : gb;
        }
      }
      __syncwarp();
      if (lane < np) {
        const float4 c0 = sp[2 * lane], c1 = sp[2 * lane + 1];
        if (c1.w != c1.w) {
          sp[2 * lane + 1].y = 1.f / c0.x;
          sp[2 * lane + 1].z = 1.f / c0.y;
        }
      }
    } else {
      // k.q of each token, and per pair k_a.k_b and k_a.q_b
      for (int it = warp - 1; it < nt + np; it += kThreads / 32 - 1) {
        const bool pair = it >= nt;
        const int ta = pair ? 2 * (it - nt) : it;
        const float *x = kd + ta * kDK;
        const float *y0 = pair ? kd + (ta + 1) * kDK : qd + ta * kDK;
        const float *y1 = qd + (ta + 1) * kDK;
        float acc0 = 0.f, acc1 = 0.f;
        for (int c = lane; c < kDK; c += 32) {
          acc0 = fmaf(x[c], y0[c], acc0);
          if (pair) acc1 = fmaf(x[c], y1[c], acc1);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          acc0 += __shfl_xor_sync(0xffffffffu, acc0, m);
          acc1 += __shfl_xor_sync(0xffffffffu, acc1, m);
        }
        if (lane == 0) {
          if (pair) gr[it - nt] = make_float2(acc0, acc1);
          else kq_s(bsel)[it] = acc0;
        }
      }
    }
    __syncthreads();
    const float *kq = kq_s(bsel);
    // odd lanes form their q products in the slots of the k products
    const float *x0 = odd ? qd : kd, *x1 = odd ? kd : qd;
    auto load_x = [&](int tt, uint64_t *xa, uint64_t *xb) {
      const ulonglong2 a0 = *reinterpret_cast<const ulonglong2 *>(x0 + tt * kDK + 4 * lc);
      const ulonglong2 a1 = *reinterpret_cast<const ulonglong2 *>(x0 + tt * kDK + 64 + 4 * lc);
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2 *>(x1 + tt * kDK + 4 * lc);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2 *>(x1 + tt * kDK + 64 + 4 * lc);
      xa[0] = a0.x; xa[1] = a0.y; xa[2] = a1.x; xa[3] = a1.y;
      xb[0] = b0.x; xb[1] = b0.y; xb[2] = b1.x; xb[3] = b1.y;
    };
    // both tokens' dot products with the state before the pair, one token at
    // a time (the state's 64 registers leave no room for both tokens' inputs
    // and products at once); returns this lane's reduced value and the
    // token's k columns
    auto dots = [&](int tt, uint64_t *kc) {
      uint64_t xa[4], xb[4];
      load_x(tt, xa, xb);
      float v[16];  // local index 2 slot + {0: xa, 1: xb}
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        v[2 * r] = dot8(S[r], xa);
        v[2 * r + 1] = dot8(S[r], xb);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) kc[q] = odd ? xb[q] : xa[q];
      float v8[8], v4[4], v2[2], v1[1];
      reduce_half<16>(v, v8, 8);
      reduce_half<8>(v8, v4, 4);
      reduce_half<4>(v4, v2, 2);
      reduce_half<2>(v2, v1, 1);
      return v1[0];
    };
    for (int pp = 0; pp < np; ++pp) {
      const int ta = 2 * pp, tb2 = ta + 1;
      uint64_t ka[4], kb[4];  // k of tokens a and b
      float a1[1], b1[1];
      a1[0] = dots(ta, ka);
      b1[0] = dots(tb2, kb);
      // even lanes: u-hat of my_row for a and b (b against the old state);
      // odd lanes: the w-hats
      const float4 c0 = sp[2 * pp], c1 = sp[2 * pp + 1];
      const float2 g = gr[pp];  // k_a.k_b, k_a.q_b
      const float vra = my_row < dv ? vd[ta * dv + my_row] : 0.f;
      const float vrb = my_row < dv ? vd[tb2 * dv + my_row] : 0.f;
      const float da = c0.z * (vra - c0.x * a1[0]);
      const float ub = fmaf(c0.x, b1[0], da * g.x);  // token b's prediction after a's update
      const float db = c0.w * (vrb - c1.x * ub);
      const float da_row = __shfl_xor_sync(0xffffffffu, da, 1);  // odd lanes: their row's d's
      const float db_row = __shfl_xor_sync(0xffffffffu, db, 1);
      if (odd && my_row < dv) {
        float *o = p.out + ((int64_t)(tb + ta) * p.Hv + h) * dv + my_row;
        o[0] = fmaf(c0.x, a1[0], da_row * kq[ta]);
        if (tb2 < nt)
          o[(int64_t)p.Hv * dv] = fmaf(c0.y, b1[0], fmaf(c1.x * da_row, g.y, db_row * kq[tb2]));
      }
      if (c1.w == c1.w) {  // fold the scale into Shat (uniform over the CTA)
        const uint64_t g2 = f2_pack(c1.w, c1.w);
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int q = 0; q < 4; ++q) S[r][q] = f2_mul(S[r][q], g2);
      }
      const float ea = da * c1.y, eb = db * c1.z;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int src = gbase + 2 * (r ^ rb);  // the lane holding slot r's row
        const float era = __shfl_sync(0xffffffffu, ea, src);
        const float erb = __shfl_sync(0xffffffffu, eb, src);
        const uint64_t ea2 = f2_pack(era, era), eb2 = f2_pack(erb, erb);
#pragma unroll
        for (int q = 0; q < 4; ++q) S[r][q] = f2_fma(eb2, kb[q], f2_fma(ea2, ka[q], S[r][q]));
      }
    }
    __syncthreads();  // the next iteration refills this buffer
  }
  cp_async_wait<0>();
  // gamma is tracked by lane 0 of warp 0
  if (tid == 0) s_gam = gam;
  __syncthreads();
  gam = s_gam;

  // final state = gamma * Shat
  TS *Sd = state_ptr();
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int row = row0 + (r ^ rb);
    if (row >= dv) continue;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int c0 = (lc + 16 * u) * 4;
      float f[4];
      f2_unpack(S[r][2 * u], f[0], f[1]);
      f2_unpack(S[r][2 * u + 1], f[2], f[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = gam * f[e];
        if constexpr (sizeof(TS) == 4) ((float *)Sd)[(int64_t)row * kDK + c0 + e] = v;
        else ((uint16_t *)Sd)[(int64_t)row * kDK + c0 + e] = float_to_bf16_bits(v);
      }
    }
  }
}

template <typename TS>
int launch_rec128_t(const RecurrentParams &p, cudaStream_t s) {
  const int64_t smem = rec128_smem_bytes(p.dv);
  static SmemLimit limit;  // per instantiation and device
  if (limit.ensure((const void *)recurrent128_kernel<TS>, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  recurrent128_kernel<TS><<<dim3(p.Hv, p.n_seq, 1), kThreads, (size_t)smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace

int launch_recurrent128(const RecurrentParams &p, int ssm_dtype, cudaStream_t s) {
  if (p.dv > kMaxDv || p.dv < 1) return LSC_ERR_UNSUPPORTED;
  return ssm_dtype == LSC_BF16 ? launch_rec128_t<__nv_bfloat16>(p, s) : launch_rec128_t<float>(p, s);
}

}  // namespace lsc
