// lsc_prefill.cu -- the prefill conv of a resumed prefill: a depthwise causal
// conv over each sequence's tokens that starts from the slot's conv state,
// the q | k | v split with the per-head L2 norm of q and k, and the write-back
// of the new conv state.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (causal_conv1d_fn beside causal_conv1d_update)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "相同前缀不一定能全部复用"
//        (the prefill continues from the restored checkpoint)
//
// The conv state of channel c holds its last W-1 inputs, oldest first.  Token
// t of a sequence sees the window [x_(t-W+1) .. x_t]; window inputs before the
// sequence's first token are the slot's conv state (zero when cold).
// y = SiLU(sum_j w[c][j] window[j]), no bias.  Afterwards the slot holds the last
// W-1 entries of [old state, the sequence's x].
//
// Kernels (one stream, in order):
//   prefill_conv_vec_kernel  (fast path) thread = 8 consecutive channels over a
//       tile of kPrefillTile tokens of the flattened token axis, rolling the
//       window in registers; each thread streams its x rows through a
//       128-byte cp.async ring in shared memory (7 bf16 or 3 f32 rows in
//       flight per thread without holding registers); the
//       sum of squares of a q/k head is reduced over the head's dk/8 lanes with
//       shuffles, so q and k leave normalised.  HBM-bound: per token and channel
//       one conv-dtype read and one fp32 write.
//   prefill_conv_scalar_kernel + qk_norm_kernel  (any other shape) one channel
//       per thread, then q and k normalised in a second pass.
//   prefill_state_kernel  the new conv state of each sequence (after the
//       outputs, so no tile reads a state another tile has already replaced).
#include <type_traits>

#include "lsc_gdn_common.cuh"

namespace lsc {
namespace {

constexpr int kPrefillThreads = 256;
constexpr int kPrefillTile = 64;  // tokens per CTA
constexpr int kPrefillRingBytes = 128;  // per thread: the cp.async ring of x rows in shared memory

// The sequence holding token t: the largest s with cu[s] <= t.  Well defined for
// consistent cu_seqlens; for others the caller checks the result.
__device__ __forceinline__ int seq_of(const int32_t *cu, int n_seq, int t) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Eight floats, passed by value.
struct F8 {
  float v[8];
};

// Eight consecutive conv-dtype values at a 16-byte-aligned address, as floats.
template <typename TC> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  __device__ __forceinline__ static F8 load(const void *p) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    F8 f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f.v[2 * i] = __uint_as_float(w[i] << 16);
      f.v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    return f;
  }
};
template <> struct Vec8<float> {
  __device__ __forceinline__ static F8 load(const void *p) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    F8 f;
    f.v[0] = a.x; f.v[1] = a.y; f.v[2] = a.z; f.v[3] = a.w;
    f.v[4] = b.x; f.v[5] = b.y; f.v[6] = b.z; f.v[7] = b.w;
    return f;
  }
};

__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Where channel c's output goes: q [T, Hk dk], k [T, Hk dk] or v [T, Hv dv].
__device__ __forceinline__ float *out_ptr(const PrefillConvParams &p, int64_t t, int c) {
  const int qk = p.Hk * p.dk;
  if (c < qk) return p.q + t * qk + c;
  if (c < 2 * qk) return p.k + t * qk + (c - qk);
  return p.v + t * (int64_t)(p.Hv * p.dv) + (c - 2 * qk);
}

// Is token t inside sequence s, with consistent bounds?  Reports otherwise.
__device__ __forceinline__ bool seq_ok(const PrefillConvParams &p, int s, int t, int &ts, int &te) {
  ts = p.cu[s];
  te = p.cu[s + 1];
  const bool ok = ts >= 0 && te >= ts && te <= p.total_tokens && ts <= t && t < te;
  if (!ok) report(p.status, LSC_ERR_INVALID_ARG);
  return ok;
}

// ------------------------------------------------------------------ fast path
// 2^x and 1/x on the special-function unit (PTX ex2.approx / rcp.approx with
// flush to zero; a few ulp of relative error each).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SiLU of a float pair: z * sigmoid(z) with sigmoid(z) = 1 / (1 + 2^(-z log2 e)).
// Large negative z gives 2^(+inf) = inf, 1/inf = 0 and SiLU -0.
__device__ __forceinline__ uint64_t silu2(uint64_t z) {
  const uint64_t neg_log2e = f2_pack(-1.44269504088896341f, -1.44269504088896341f);
  const uint64_t one = f2_pack(1.f, 1.f);
  float a, b;
  f2_unpack(f2_mul(z, neg_log2e), a, b);
  f2_unpack(f2_add(f2_pack(ex2_approx(a), ex2_approx(b)), one), a, b);
  return f2_mul(z, f2_pack(rcp_approx(a), rcp_approx(b)));
}

// Eight consecutive conv-dtype values at a 16-byte-aligned global address, as
// four float pairs (channel 2i low, 2i + 1 high).
template <typename TC>
__device__ __forceinline__ void load_pairs8(const void *p, uint64_t *f) {
  const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
  for (int h = 0; h < 8 * (int)sizeof(TC) / 16; ++h) StatePairs<TC>::unpack(__ldg(q + h), f + h * StatePairs<TC>::N);
}

template <int R>
using Rot = std::integral_constant<int, R>;

// Calls tok(Rot<R>{}) for R = R0 .. H-1, one token each, advancing t; false
// once t reaches end.
template <int R, int H, typename F>
__device__ __forceinline__ bool tokens_rotated(F &tok, int &t, int end) {
  if constexpr (R == H) {
    return true;
  } else {
    tok(Rot<R>{});
    if (++t >= end) return false;
    return tokens_rotated<R + 1, H>(tok, t, end);
  }
}

// Every kernel of this file is launched with programmatic stream
// serialisation (launch_pdl): it waits here, before any global access, for the
// kernel before it on the stream to complete, then lets the next be placed.
__device__ __forceinline__ void pdl_enter() {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
}

template <typename TC, int CW>
__global__ void __launch_bounds__(kPrefillThreads, CW ? 3 : 1) prefill_conv_vec_kernel(const __grid_constant__ PrefillConvParams p) {
  pdl_enter();
  constexpr int WW = CW ? CW : kMaxTaps;  // register window, W <= WW
  constexpr int H = WW - 1;               // window inputs before the current token
  constexpr int esc = (int)sizeof(TC);
  const int W = CW ? CW : p.conv_width;
  const int C = p.conv_dim;
  const int grp = blockIdx.x * kPrefillThreads + threadIdx.x;
  const bool live = grp < C / 8;
  const int c0 = live ? grp * 8 : 0;
  const int lanes_per_head = p.dk / 8;  // a power of two <= 32
  const int qk = p.Hk * p.dk;
  const bool is_qk = live && c0 < 2 * qk;
  const int t_begin = blockIdx.y * kPrefillTile;
  const int t_end = min(t_begin + kPrefillTile, p.total_tokens);
  if (t_begin >= t_end) return;  // uniform over the CTA
  // does any lane of the warp carry q or k channels (the norm's shuffles then
  // run on the whole warp)
  const bool warp_qk = __any_sync(0xffffffffu, is_qk);

  __shared__ int s_first;
  if (threadIdx.x == 0) s_first = seq_of(p.cu, p.n_seq, t_begin);
  __syncthreads();

  // where the group's outputs go: q [T, Hk dk], k [T, Hk dk] or v [T, Hv dv]
  float *obase;
  int64_t orow;
  if (c0 < qk) {
    obase = p.q + c0;
    orow = qk;
  } else if (c0 < 2 * qk) {
    obase = p.k + (c0 - qk);
    orow = qk;
  } else {
    obase = p.v + (c0 - 2 * qk);
    orow = (int64_t)p.Hv * p.dv;
  }

  // weights of the group's 8 channels as pairs: w2[i][j] = tap j of channels 2i, 2i + 1
  uint64_t w2[4][WW];
  {
    F8 buf[WW];  // the 8 W weights of the group, row-major [8][W]
    const uint8_t *wp = reinterpret_cast<const uint8_t *>(p.w) + (int64_t)c0 * W * esc;
#pragma unroll
    for (int v = 0; v < WW; ++v) buf[v] = v < W ? Vec8<TC>::load(wp + v * 8 * esc) : F8{};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < WW; ++j) {
        float wv[2] = {0.f, 0.f};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 8 * WW; ++e)
            if (e == (2 * i + h) * W + j && j < W) wv[h] = buf[e / 8].v[e % 8];
        w2[i][j] = f2_pack(wv[0], wv[1]);
      }
  }
  const uint8_t *xg = reinterpret_cast<const uint8_t *>(p.x) + (int64_t)c0 * esc;
  const int64_t xrow = (int64_t)C * esc;

  constexpr int NH = 8 * esc / 16;  // 16-byte pieces of one x row of the group
  constexpr int A = kPrefillRingBytes / (8 * esc);  // ring slots: 8 rows (bf16) or 4 (f32)
  __shared__ __align__(16) uint4 ring[A][NH][kPrefillThreads];
  // hist[(j + R) % H] is window input j (0 = oldest) of a token processed at
  // rotation R: a new token's x overwrites the oldest input in place.  With a
  // run-time width (CW = 0) the rotation stays 0 and the inputs shift instead.
  uint64_t hist[H][4];
  int s = s_first;
  // The tile is walked in segments, one per sequence piece: the window is
  // rebuilt at a segment's first token, then slides token by token.
  for (int t = t_begin; t < t_end;) {
    while (s + 1 < p.n_seq && p.cu[s + 1] <= t) ++s;
    int ts, te;
    const bool ok = seq_ok(p, s, t, ts, te);
    const int seg_end = ok ? min(te, t_end) : t + 1;  // a bad sequence is re-checked token by token
    int32_t slot = ok ? p.idx[s] : -1;
    if (slot >= p.num_slots) {
      report(p.status, LSC_ERR_OUT_OF_RANGE);
      slot = -1;
    }
    const bool warm = slot >= 0 && (p.has_init == nullptr || p.has_init[s] != 0);
    {
      F8 st[H];  // the group's conv state, row-major [8][W - 1]
#pragma unroll
      for (int v = 0; v < H; ++v) st[v] = F8{};
      if (warm && live && t - ts < W - 1) {
        const uint8_t *sp = p.layer + (int64_t)slot * p.page + (int64_t)c0 * (W - 1) * esc;
#pragma unroll
        for (int v = 0; v < H; ++v)
          if (v < W - 1) st[v] = Vec8<TC>::load(sp + v * 8 * esc);
      }
      // window input j is token t - (W - 1 - j); before the sequence it is
      // state entry (t - ts) + j (entries are picked with compile-time indices)
#pragma unroll
      for (int j = 0; j < H; ++j) {
        if (j >= W - 1) continue;
        const int back = W - 1 - j;
        if (t - back >= ts) {
          load_pairs8<TC>(xg + (int64_t)(t - back) * xrow, hist[j]);
        } else {
          const int e = (t - ts) + j;
          float val[8];
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            val[cc] = 0.f;
#pragma unroll
            for (int ee = 0; ee < 8 * H; ++ee)
              if (ee == cc * (W - 1) + e) val[cc] = st[ee / 8].v[ee % 8];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) hist[j][i] = f2_pack(val[2 * i], val[2 * i + 1]);
        }
      }
    }
    // the ring: slot (u % A) holds token seg_t0 + u.  One cp.async group per
    // token (empty past the segment).  Token u + A - 1 is issued into the slot
    // read one token earlier, then wait_group<A - 1> leaves token u landed.
    const int seg_t0 = t;
#pragma unroll
    for (int u = 0; u < A - 1; ++u) {
      if (seg_t0 + u < seg_end)
#pragma unroll
        for (int h = 0; h < NH; ++h)
          cp_async16(&ring[u][h][threadIdx.x], xg + (int64_t)(seg_t0 + u) * xrow + h * 16);
      cp_async_commit();
    }
    auto token = [&](auto rot) {
      constexpr int R = decltype(rot)::value;
      const int u = t - seg_t0;
      if (t + A - 1 < seg_end)
#pragma unroll
        for (int h = 0; h < NH; ++h)
          cp_async16(&ring[(u + A - 1) % A][h][threadIdx.x], xg + (int64_t)(t + A - 1) * xrow + h * 16);
      cp_async_commit();
      cp_async_wait<A - 1>();
      uint64_t xc[4];
#pragma unroll
      for (int h = 0; h < NH; ++h) StatePairs<TC>::unpack(ring[u % A][h][threadIdx.x], xc + h * StatePairs<TC>::N);
      uint64_t y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint64_t z = f2_mul(w2[i][0], hist[R % H][i]);  // W >= 2: tap 0 is a window input
#pragma unroll
        for (int j = 1; j < WW; ++j) {
          if (j < W - 1) z = f2_fma(w2[i][j], hist[(j + R) % H][i], z);
          else if (j == W - 1) z = f2_fma(w2[i][j], xc[i], z);
        }
        y[i] = silu2(z);
      }
      // slide the window: this token's x replaces the oldest input
      if constexpr (CW != 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) hist[R % H][i] = xc[i];
      } else {
#pragma unroll
        for (int j = 0; j < H - 1; ++j)
          if (j < W - 2)
#pragma unroll
            for (int i = 0; i < 4; ++i) hist[j][i] = hist[j + 1][i];
#pragma unroll
        for (int j = 0; j < H; ++j)
          if (j == W - 2)
#pragma unroll
            for (int i = 0; i < 4; ++i) hist[j][i] = xc[i];
      }
      // q and k: divide by the head's sqrt(sum of squares + 1e-6); the head's
      // dk/8 lanes are consecutive and aligned, reduced with shuffles
      float scale = 1.f;
      if (warp_qk) {
        uint64_t s2 = f2_mul(y[0], y[0]);
#pragma unroll
        for (int i = 1; i < 4; ++i) s2 = f2_fma(y[i], y[i], s2);
        float a, b;
        f2_unpack(s2, a, b);
        float ss = a + b;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1)
          if (m < lanes_per_head) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (is_qk) scale = rsqrtf(ss + 1e-6f);
      }
      if (live) {
        float4 *o = reinterpret_cast<float4 *>(obase + (int64_t)t * orow);
        if (slot >= 0) {
          const uint64_t sc = f2_pack(scale, scale);
          float f[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) f2_unpack(warp_qk ? f2_mul(y[i], sc) : y[i], f[2 * i], f[2 * i + 1]);
          o[0] = make_float4(f[0], f[1], f[2], f[3]);
          o[1] = make_float4(f[4], f[5], f[6], f[7]);
        } else {
          o[0] = o[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    };
    if constexpr (CW != 0) {
      while (t < seg_end && tokens_rotated<0, H>(token, t, seg_end)) {
      }
    } else {
      for (; t < seg_end; ++t) token(Rot<0>{});
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- any shape
template <typename TC>
__global__ void __launch_bounds__(kPrefillThreads) prefill_conv_scalar_kernel(const __grid_constant__ PrefillConvParams p) {
  pdl_enter();
  using E = Elem<TC>;
  const int W = p.conv_width, C = p.conv_dim;
  const int c = blockIdx.x * kPrefillThreads + threadIdx.x;
  const bool live = c < C;
  const int t_begin = blockIdx.y * kPrefillTile;
  const int t_end = min(t_begin + kPrefillTile, p.total_tokens);
  if (t_begin >= t_end) return;
  __shared__ int s_first;
  if (threadIdx.x == 0) s_first = seq_of(p.cu, p.n_seq, t_begin);
  __syncthreads();
  if (!live) return;
  float wt[kMaxTaps], hist[kMaxTaps - 1];
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j) wt[j] = j < W ? E::ld(p.w, (int64_t)c * W + j) : 0.f;
  int s = s_first, ts = 0, te = 0;
  int32_t slot = -1;
  for (int t = t_begin; t < t_end; ++t) {
    if (t == t_begin || t >= te) {
      while (s + 1 < p.n_seq && p.cu[s + 1] <= t) ++s;
      const bool ok = seq_ok(p, s, t, ts, te);
      slot = ok ? p.idx[s] : -1;
      if (slot >= p.num_slots) {
        report(p.status, LSC_ERR_OUT_OF_RANGE);
        slot = -1;
      }
      if (!ok) te = t + 1;
      const bool warm = slot >= 0 && (p.has_init == nullptr || p.has_init[s] != 0);
      const uint8_t *sp = slot >= 0 ? p.layer + (int64_t)slot * p.page : nullptr;
#pragma unroll
      for (int j = 0; j < kMaxTaps - 1; ++j) {
        if (j >= W - 1) continue;
        const int back = W - 1 - j;  // hist[j] is token t - back
        hist[j] = t - back >= ts ? E::ld(p.x, (int64_t)(t - back) * C + c)
                                 : (warm ? E::ld(sp, (int64_t)c * (W - 1) + (t - ts) + j) : 0.f);
      }
    }
    const float xc = E::ld(p.x, (int64_t)t * C + c);
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTaps; ++j) {
      if (j < W - 1) z = fmaf(wt[j], hist[j], z);
      else if (j == W - 1) z = fmaf(wt[j], xc, z);
    }
#pragma unroll
    for (int j = 0; j < kMaxTaps - 1; ++j) {
      if (j < W - 2) hist[j] = hist[j + 1 < kMaxTaps - 1 ? j + 1 : j];
      else if (j == W - 2) hist[j] = xc;
    }
    *out_ptr(p, t, c) = slot >= 0 ? silu(z) : 0.f;
  }
}

// q and k of every (token, head) divided by sqrt(sum of squares + 1e-6): one
// warp per (token, head).
__global__ void __launch_bounds__(kPrefillThreads) qk_norm_kernel(const __grid_constant__ PrefillConvParams p) {
  pdl_enter();
  const int64_t wid = (int64_t)blockIdx.x * (kPrefillThreads / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)p.total_tokens * p.Hk * 2;
  if (wid >= n) return;
  const int64_t th = wid / 2;  // (token, head)
  float *base = ((wid & 1) ? p.k : p.q) + th * p.dk;
  float ss = 0.f;
  for (int c = lane; c < p.dk; c += 32) ss = fmaf(base[c], base[c], ss);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
  const float inv = 1.f / sqrtf(ss + 1e-6f);
  for (int c = lane; c < p.dk; c += 32) base[c] *= inv;
}

// The new conv state of each sequence: the last W-1 entries of [old state, x],
// copied bit for bit.  One thread per (sequence, channel).
template <typename TB>  // raw element bits: uint16_t (bf16) or uint32_t (f32)
__global__ void __launch_bounds__(kPrefillThreads) prefill_state_kernel(const __grid_constant__ PrefillConvParams p) {
  pdl_enter();  // the conv kernel before it has read every old conv state
  const int W = p.conv_width, C = p.conv_dim;
  const int c = blockIdx.x * kPrefillThreads + threadIdx.x;
  const int s = blockIdx.y;
  if (c >= C) return;
  const int ts = p.cu[s], te = p.cu[s + 1];
  if (ts < 0 || te < ts || te > p.total_tokens) {  // inconsistent cu_seqlens: touch nothing
    if (c == 0) report(p.status, LSC_ERR_INVALID_ARG);
    return;
  }
  const int32_t slot = p.idx[s];
  if (slot < 0 || slot >= p.num_slots) return;
  const bool warm = p.has_init == nullptr || p.has_init[s] != 0;
  TB *st = reinterpret_cast<TB *>(p.layer + (int64_t)slot * p.page) + (int64_t)c * (W - 1);
  const TB *x = reinterpret_cast<const TB *>(p.x);
  const int L = te - ts;
  TB old[kMaxTaps - 1], nv[kMaxTaps - 1];
#pragma unroll
  for (int j = 0; j < kMaxTaps - 1; ++j) old[j] = (j < W - 1 && warm) ? st[j] : TB(0);
#pragma unroll
  for (int j = 0; j < kMaxTaps - 1; ++j) {
    if (j >= W - 1) continue;
    const int pos = L - (W - 1) + j;  // position in the sequence of the entry
    nv[j] = pos >= 0 ? x[(int64_t)(ts + pos) * C + c] : old[(W - 1) + pos];
  }
#pragma unroll
  for (int j = 0; j < kMaxTaps - 1; ++j)
    if (j < W - 1) st[j] = nv[j];
}

template <typename TC>
int launch_prefill_t(const PrefillConvParams &p, cudaStream_t s) {
  const int tiles = (p.total_tokens + kPrefillTile - 1) / kPrefillTile;
  if (tiles > 0) {
    cudaError_t e;
    if (p.vec) {
      const dim3 grid((p.conv_dim / 8 + kPrefillThreads - 1) / kPrefillThreads, tiles);
      e = p.conv_width == 4 ? launch_pdl(prefill_conv_vec_kernel<TC, 4>, grid, kPrefillThreads, 0, s, p)
                            : launch_pdl(prefill_conv_vec_kernel<TC, 0>, grid, kPrefillThreads, 0, s, p);
    } else {
      const dim3 grid((p.conv_dim + kPrefillThreads - 1) / kPrefillThreads, tiles);
      e = launch_pdl(prefill_conv_scalar_kernel<TC>, grid, kPrefillThreads, 0, s, p);
      const int64_t warps = (int64_t)p.total_tokens * p.Hk * 2;
      const int64_t blocks = (warps + kPrefillThreads / 32 - 1) / (kPrefillThreads / 32);
      if (e == cudaSuccess && blocks > 0) e = launch_pdl(qk_norm_kernel, dim3((unsigned)blocks), kPrefillThreads, 0, s, p);
    }
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
  }
  if (p.n_seq > 0) {
    const dim3 grid((p.conv_dim + kPrefillThreads - 1) / kPrefillThreads, p.n_seq);
    const cudaError_t e = sizeof(TC) == 2 ? launch_pdl(prefill_state_kernel<uint16_t>, grid, kPrefillThreads, 0, s, p)
                                          : launch_pdl(prefill_state_kernel<uint32_t>, grid, kPrefillThreads, 0, s, p);
    if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
  }
  return LSC_OK;
}

}  // namespace

int launch_prefill_conv(const PrefillConvParams &p, cudaStream_t stream) {
  if (p.conv_width < 2 || p.conv_width > kMaxTaps) return LSC_ERR_UNSUPPORTED;
  return p.conv_bf16 ? launch_prefill_t<__nv_bfloat16>(p, stream) : launch_prefill_t<float>(p, stream);
}

}  // namespace lsc
