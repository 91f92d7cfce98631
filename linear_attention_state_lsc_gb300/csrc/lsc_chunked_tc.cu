// lsc_chunked_tc.cu -- the state kernel of the chunked gated delta rule on the
// 5th-generation tensor cores (tcgen05, TMEM accumulators): the resumed-prefill
// recurrence run 64 tokens at a time from the restored state, with the
// state-free quantities of every chunk (T', B, E, F, e_last; lsc_chunk.h) read
// from the workspace records that the preparation kernel (lsc_chunk_prep.cu)
// wrote before it on the same stream.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule, the token recurrence)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with
//        q); "相同前缀不一定能全部复用" (continue from the restored checkpoint)
// The pages give the token recurrence only; the chunked form is its algebraic
// rearrangement, exact up to rounding.
//
// Per chunk and v head (M 128 = state rows = TMEM lanes):
//   [P' | R'] = S [E o K; E o Q]^T    N 128, K 128   A = S from TMEM
//   D  = (V - P') T'^T                N 64,  K 64    A = X = V - P' from TMEM
//   S  = e_last S + D (F o K)         N 128, K 64    A = D from TMEM
//   O  = R' + D B^T                   N 64,  K 64    A = D from TMEM (o_t of every row)
// Products in tf32 with an fp32 accumulator.  Every operand x is split as
// x = hi + lo and each product formed as hi.hi + hi.lo + lo.hi: about 22
// significant bits per operand, so the products carry fp32-level error (the
// dropped lo.lo term is below 2^-21 of the product).  The tensor cores read a
// 32-bit operand as tf32 by truncation (its low 13 bits ignored), so the state
// in TMEM serves as its own hi part and only lo = tf32(S - trunc(S)) is
// written; the other operands use hi = tf32 rounded to nearest.
//
// CTA = one (sequence, v head), 256 threads, one CTA per SM (TMEM: all 512
// columns; shared memory ~201 KB).  Every warp runs the same code: warp w
// reaches TMEM lanes 32 (w % 4) .. + 31, so thread (w, lane) owns state row
// r = 32 (w % 4) + lane and the column half w / 4 of each row-wise pass (lo of
// S, X, the decay, the split of D, the outputs), and a share of every operand
// tile stored to shared memory.  Warp 0 waits until the operands of a product
// are in place and one elected lane issues its MMAs and commits them (from
// converged code, so the operands stay warp-uniform).  Per chunk c:
//   [P' | R'](c) on the tensor core, meanwhile F o K (c) stored -> X formed,
//   T' and B (c) stored over the [E o K; E o Q] tile -> D(c), meanwhile S
//   decayed -> D split -> O(c), then update(c), meanwhile E o K (c+1) stored
//   over T', E o Q (c+1) over B -> lo of S (c+1); the outputs of chunk c are
//   written while [P' | R'](c+1) runs.
// The loads of chunk c+1 (k, q, v, records) are issued during chunk c.
// Hand-offs go through mbarriers: threads -> MMA (operands written), MMA ->
// threads (tcgen05.commit).  Every wait is bounded: on expiry the thread
// records LSC_ERR_DEV_TIMEOUT, the CTA stops issuing work, waits (bounded)
// for the MMAs it issued and frees its TMEM.
//
// TMEM columns (lanes = state rows):
//   0-127    S (fp32; the hi part of its own split)
//   128-255  lo of S; after [P' | R']: X hi (128-191), X lo (192-255); after
//            D: D hi (128-191), D lo (192-255)
//   256-383  [P' | R'] of even chunks: P' (256-319), then D; R' (320-383), then O
//   384-511  the same for odd chunks, so that a chunk's outputs are written
//            while the next chunk's [P' | R'] runs
// Shared-memory tiles (no swizzle, lsc_chunk.h): the token-major [E o K; E o Q]
// tile (hi, lo), T' over its k half and B over its q half once [P' | R'] has
// read it; F o K channel-major (hi, lo).
#include "lsc_chunk.h"
#include "lsc_gdn_common.cuh"
#include "lsc_tc.h"

namespace lsc {
namespace {

using namespace chunk;

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t T_S = 0;
constexpr uint32_t T_LO = 128;   // lo of S; X hi / lo; D hi / lo
constexpr uint32_t T_PR = 256;   // [P' | R'] of even chunks (P', then D; R', then O); odd chunks at + 128

constexpr uint32_t OFF_KQHI = 0;
constexpr uint32_t OFF_KQLO = kKqBytes;
constexpr uint32_t OFF_KTHI = 2 * kKqBytes;
constexpr uint32_t OFF_KTLO = OFF_KTHI + kKtBytes;
constexpr uint32_t kSmemBytes = OFF_KTLO + kKtBytes;
constexpr uint32_t OFF_THI = OFF_KQHI, OFF_TLO = OFF_KQLO;                    // T' over the k half
constexpr uint32_t OFF_BHI = OFF_KQHI + kQRow0, OFF_BLO = OFF_KQLO + kQRow0;  // B over the q half
static_assert(kSmemBytes <= 226 * 1024, "shared memory budget (one CTA per SM)");

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, uint64_t limit, int32_t *status,
                                              volatile int *abort_flag) {
  if (mbar_wait_bounded(bar, parity, limit)) return true;
  report(status, LSC_ERR_DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// true on every thread of the CTA when v is true on any of them; leaves every
// warp reconverged for the warp-wide .sync.aligned TMEM loads and stores
__device__ __forceinline__ bool cta_any(bool v) {
  const bool r = __syncthreads_or(v) != 0;
  __syncwarp();
  return r;
}

struct Bars {
  uint64_t kqk, kqq, kt;   // E o K, E o Q, F o K stored (every thread)
  uint64_t split, xt, dd;  // lo of S; X, T' and B; D hi / lo and the decayed S written (every thread)
  uint64_t pr, d, u, o;    // MMA commits
};

__device__ __forceinline__ void sts_split4(uint8_t *sm, uint32_t off_hi, uint32_t off_lo, float4 f) {
  uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
  tc::split_tf32(f.x, h0, l0);
  tc::split_tf32(f.y, h1, l1);
  tc::split_tf32(f.z, h2, l2);
  tc::split_tf32(f.w, h3, l3);
  *reinterpret_cast<uint4 *>(sm + off_hi) = make_uint4(h0, h1, h2, h3);
  *reinterpret_cast<uint4 *>(sm + off_lo) = make_uint4(l0, l1, l2, l3);
}

__device__ __forceinline__ float4 ldg4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }

__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }

// 4 x 4 transpose inside each aligned group of four lanes: lane k of the
// group holds a[c] = element (k, c) and ends with a[r] = element (r, k).  Two
// exchange steps (lanes k ^ 1, then k ^ 2), two shuffles each.
__device__ __forceinline__ void transpose4(float (&a)[4], int lane) {
  const bool odd = lane & 1, high = lane & 2;
  float x0 = odd ? a[0] : a[1], x1 = odd ? a[2] : a[3];
  float y0 = __shfl_xor_sync(0xffffffffu, x0, 1), y1 = __shfl_xor_sync(0xffffffffu, x1, 1);
  const float t0 = odd ? y0 : a[0], t1 = odd ? a[1] : y0, t2 = odd ? y1 : a[2], t3 = odd ? a[3] : y1;
  x0 = high ? t0 : t2;
  x1 = high ? t1 : t3;
  y0 = __shfl_xor_sync(0xffffffffu, x0, 2);
  y1 = __shfl_xor_sync(0xffffffffu, x1, 2);
  a[0] = high ? y0 : t0;
  a[1] = high ? y1 : t1;
  a[2] = high ? t2 : y0;
  a[3] = high ? t3 : y1;
}

// lo part of x when the tensor cores read x itself as its hi part (truncation)
__device__ __forceinline__ uint32_t lo_of_truncated(float x) {
  return tc::to_tf32(x - __uint_as_float(__float_as_uint(x) & 0xffffe000u));
}

// ---- MMA issue (one thread; three tf32 passes per product) --------------------
// A from TMEM (hi at a_hi, lo at a_lo; a k step of 8 columns), B from a
// K-major shared-memory tile (hi / lo descriptors; a k step advances the start
// address by kstep16 16-byte units).
template <int KSTEPS>
__device__ __forceinline__ void issue3(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint64_t b_hi, uint64_t b_lo,
                                       uint32_t kstep16, uint32_t idesc, bool acc) {
#pragma unroll
  for (int ps = 0; ps < 3; ++ps) {
    const uint32_t a = ps == 2 ? a_lo : a_hi;
    const uint64_t b = ps == 1 ? b_lo : b_hi;
#pragma unroll
    for (int k = 0; k < KSTEPS; ++k)
      tc::mma_ts(d, a + 8 * k, b + (uint64_t)(kstep16 * k), idesc, (acc || ps != 0 || k != 0) ? 1u : 0u);
  }
}

template <typename TS>
__global__ void __launch_bounds__(kThreads, 1) chunked_tc_kernel(const __grid_constant__ RecurrentParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int32_t s_len[kRankedSeqs];
  __shared__ int32_t s_seq;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, g = h / p.group;
  const int dv = p.dv;

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
  const int nch = (t1 - t0 + kC - 1) / kC;
  // record of chunk c: recs + c * rec_stride
  const float *recs = p.ws + (slot_base(t0, i) * p.Hv + h) * (int64_t)kRecFloats;
  const int64_t rec_stride = (int64_t)p.Hv * kRecFloats;
  TS *Sg = reinterpret_cast<TS *>(p.layer + (int64_t)slot * p.page + p.ssm_off) + (int64_t)h * dv * kDK;

  if (tid == 0) {
    mbar_init(&bars.kqk, kThreads);
    mbar_init(&bars.kqq, kThreads);
    mbar_init(&bars.kt, kThreads);
    mbar_init(&bars.split, kThreads);
    mbar_init(&bars.xt, kThreads);
    mbar_init(&bars.dd, kThreads);
    mbar_init(&bars.pr, 1);
    mbar_init(&bars.d, 1);
    mbar_init(&bars.u, 1);
    mbar_init(&bars.o, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 0) {
    __syncwarp();
    tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  volatile int *abort_flag = &s_abort;
  const uint64_t lim = p.wait_limit_ns;

  // this thread's state row, column half and TMEM lanes
  const int r0 = 32 * (warp & 3), r = r0 + lane, hf = warp >> 2;
  // v and out move as 16-byte pieces (four rows of a token) when their rows
  // allow it; lane 4 q + k then reaches rows r0 + 4 q .. + 3 of token 4 i + k
  const bool vec = dv % 4 == 0 && (((uintptr_t)p.v | (uintptr_t)p.out) & 15) == 0;
  const int rq = r0 + 4 * (lane >> 2), kq = lane & 3;
  const bool row_ok = r < dv;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  // operand tiles: k / q blocks (tokens 4a..4a+3, a = al + 8 ah; channels
  // 4 cg..4 cg+3) and T' / B pieces (row trow, columns 16 q4 + 4 m)
  const int al = lane & 7, cg = (lane >> 3) + 4 * warp;
  const int trow = tid & 63, q4 = tid >> 6;

  constexpr uint32_t id64 = tc::idesc_tf32(128, 64, false);
  constexpr uint32_t id128 = tc::idesc_tf32(128, 128, false);
  // B operand descriptors; a k step of 8 tf32 columns is 256 bytes along the
  // token-major tile, 2 kLbo bytes along a 64-column tile
  const uint64_t dkq_hi = tc::smem_desc(smem_u32(sm + OFF_KQHI), 128, kKqRg);
  const uint64_t dkq_lo = tc::smem_desc(smem_u32(sm + OFF_KQLO), 128, kKqRg);
  const uint64_t dt_hi = tc::smem_desc(smem_u32(sm + OFF_THI), kLbo, kRg64);
  const uint64_t dt_lo = tc::smem_desc(smem_u32(sm + OFF_TLO), kLbo, kRg64);
  const uint64_t db_hi = tc::smem_desc(smem_u32(sm + OFF_BHI), kLbo, kRg64);
  const uint64_t db_lo = tc::smem_desc(smem_u32(sm + OFF_BLO), kLbo, kRg64);
  const uint64_t dkt_hi = tc::smem_desc(smem_u32(sm + OFF_KTHI), kLbo, kRg64);
  const uint64_t dkt_lo = tc::smem_desc(smem_u32(sm + OFF_KTLO), kLbo, kRg64);
  constexpr uint32_t kq_step = 256 >> 4, sq_step = (2 * kLbo) >> 4;
  uint64_t *last = nullptr;  // warp 0: the last commit's barrier and phase
  uint32_t last_par = 0;

  // ---- per-chunk operands held in registers ----------------------------------
  float4 kr[2][4], qr[2][4];  // k, q of this thread's blocks
  float ev[2][4], fv[2][4];   // E, F of its tokens
  float4 tv[4], bv[4];        // T', B pieces
  float x[32];                // v of its row at tokens 32 hf .. 32 hf + 31 (vec: before transposing)
  float e_last = 1.f;
  auto load_kq = [&](int c) {
    const int nt = min(kC, t1 - t0 - c * kC);
    const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
    const float *rec = recs + c * rec_stride;
#pragma unroll
    for (int ah = 0; ah < 2; ++ah) {
      const float4 e4 = ldg4(rec + kRecE + 4 * (al + 8 * ah)), f4 = ldg4(rec + kRecF + 4 * (al + 8 * ah));
      ev[ah][0] = e4.x, ev[ah][1] = e4.y, ev[ah][2] = e4.z, ev[ah][3] = e4.w;
      fv[ah][0] = f4.x, fv[ah][1] = f4.y, fv[ah][2] = f4.z, fv[ah][3] = f4.w;
    }
#pragma unroll
    for (int ah = 0; ah < 2; ++ah)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tok = 4 * (al + 8 * ah) + u;
        const int64_t off = ((tb + tok) * p.Hk + g) * kDK + 4 * cg;
        const bool in = tok < nt;
        kr[ah][u] = in ? ldg4(p.k + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        qr[ah][u] = in ? ldg4(p.q + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
  };
  auto load_rest = [&](int c) {  // v, T', B and e_last of chunk c
    const int nt = min(kC, t1 - t0 - c * kC);
    const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
    const float *rec = recs + c * rec_stride;
    if (vec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = 32 * hf + 4 * i + kq;
        const float4 f =
            (t < nt && rq < dv) ? ldg4(p.v + ((tb + t) * p.Hv + h) * dv + rq) : make_float4(0.f, 0.f, 0.f, 0.f);
        x[4 * i] = f.x, x[4 * i + 1] = f.y, x[4 * i + 2] = f.z, x[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int t = 32 * hf + e;
        x[e] = (t < nt && row_ok) ? __ldg(p.v + ((tb + t) * p.Hv + h) * dv + r) : 0.f;
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j4 = 16 * q4 + 4 * m;
      const bool in = j4 < 4 * row_groups(trow);
      tv[m] = in ? ldg4(rec + kRecT + rec_off(trow, j4)) : make_float4(0.f, 0.f, 0.f, 0.f);
      bv[m] = in ? ldg4(rec + kRecB + rec_off(trow, j4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    e_last = __ldg(rec + kRecMisc);
  };
  // token-major E o K (rows 0-63) or E o Q (rows 64-127)
  auto store_rows = [&](const float4 (&src)[2][4], int row0) {
#pragma unroll
    for (int ah = 0; ah < 2; ++ah)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = row0 + 4 * (al + 8 * ah) + u;
        sts_split4(sm, OFF_KQHI + kq_off(j, 4 * cg), OFF_KQLO + kq_off(j, 4 * cg), scale4(src[ah][u], ev[ah][u]));
      }
  };
  // channel-major F o K: K[j][c] F_j at (channel c, token j)
  auto store_kt = [&]() {
#pragma unroll
    for (int ah = 0; ah < 2; ++ah) {
      const int a = al + 8 * ah;
      const float4 *k4 = kr[ah];
      const float f0 = fv[ah][0], f1 = fv[ah][1], f2 = fv[ah][2], f3 = fv[ah][3];
      const float col[4][4] = {{k4[0].x * f0, k4[1].x * f1, k4[2].x * f2, k4[3].x * f3},
                               {k4[0].y * f0, k4[1].y * f1, k4[2].y * f2, k4[3].y * f3},
                               {k4[0].z * f0, k4[1].z * f1, k4[2].z * f2, k4[3].z * f3},
                               {k4[0].w * f0, k4[1].w * f1, k4[2].w * f2, k4[3].w * f3}};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ch = 4 * cg + e;
        sts_split4(sm, OFF_KTHI + sq_off(ch, 4 * a), OFF_KTLO + sq_off(ch, 4 * a),
                   make_float4(col[e][0], col[e][1], col[e][2], col[e][3]));
      }
    }
  };
  auto publish = [&](uint64_t *bar) {
    fence_proxy_async_smem();  // generic-proxy stores, read by the MMA
    mbar_arrive(bar);
  };
  // lo of S (this thread's 64 columns) -> TMEM, then arrive on `split`
  auto split_state = [&]() {
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      uint32_t v[32];
      tc::tmem_ld32(tl + T_S + 64 * hf + 32 * q, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = lo_of_truncated(__uint_as_float(v[e]));
      tc::tmem_st32(tl + T_LO + 64 * hf + 32 * q, v);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    mbar_arrive(&bars.split);
  };
  // outputs of chunk c: O columns 32 hf .. + 31 of this row (buffer c % 2)
  auto write_out = [&](int c) {
    const int nt = min(kC, t1 - t0 - c * kC);
    const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
    uint32_t w[32];
    tc::tmem_ld32(tl + T_PR + 128 * (c & 1) + 64 + 32 * hf, w);
    tc::tmem_wait_ld();
    if (vec) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float a[4] = {__uint_as_float(w[4 * i]), __uint_as_float(w[4 * i + 1]), __uint_as_float(w[4 * i + 2]),
                      __uint_as_float(w[4 * i + 3])};
        transpose4(a, lane);  // lane 4 q + k: rows rq .. rq + 3 of token 4 i + k
        const int t = 32 * hf + 4 * i + kq;
        if (t < nt && rq < dv)
          *reinterpret_cast<float4 *>(p.out + ((tb + t) * p.Hv + h) * dv + rq) = make_float4(a[0], a[1], a[2], a[3]);
      }
    } else if (row_ok) {
      float *o = p.out + ((tb + 32 * hf) * p.Hv + h) * dv + r;
      const int64_t ostride = (int64_t)p.Hv * dv;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (32 * hf + e < nt) o[e * ostride] = __uint_as_float(w[e]);
    }
  };

  // ---- initial state -> TMEM (zero when cold; rows >= dv stay zero)
#pragma unroll 1
  for (int q = 0; q < 2; ++q) {
    uint32_t v[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = 0u;
    const int col0 = 64 * hf + 32 * q;
    if (warm && row_ok) {
      if constexpr (sizeof(TS) == 4) {
        const float4 *src = reinterpret_cast<const float4 *>(Sg + (int64_t)r * kDK + col0);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 f = __ldg(src + e);
          v[4 * e] = __float_as_uint(f.x);
          v[4 * e + 1] = __float_as_uint(f.y);
          v[4 * e + 2] = __float_as_uint(f.z);
          v[4 * e + 3] = __float_as_uint(f.w);
        }
      } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(Sg + (int64_t)r * kDK + col0);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 b = __ldg(src + e);
          const uint32_t w4[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * e + 2 * k] = w4[k] << 16;
            v[8 * e + 2 * k + 1] = w4[k] & 0xffff0000u;
          }
        }
      }
    }
    __syncwarp();
    tc::tmem_st32(tl + T_S + col0, v);
  }
  tc::tmem_wait_st();

  // ---- chunk 0's operands
  if (nch > 0) {
    load_kq(0);
    load_rest(0);
    split_state();
    store_rows(kr, 0);
    publish(&bars.kqk);
    store_rows(qr, kC);
    publish(&bars.kqq);
    store_kt();
    publish(&bars.kt);
  }

  bool ok = true;
#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const uint32_t par = c & 1;
    const uint32_t pr = T_PR + 128 * par;  // this chunk's [P' | R'] buffer
    const bool more = c + 1 < nch;
    bool ok0 = true;  // warp 0: its waits succeeded
    // ---- [P' | R'] once lo of S and the [E o K; E o Q] tile are in place
    if (warp == 0) {
      // every lane observes the operands' barriers (the elected lane issues)
      ok0 = wait_or_abort(&bars.split, par, lim, p.status, abort_flag) &&
            wait_or_abort(&bars.kqk, par, lim, p.status, abort_flag) &&
            wait_or_abort(&bars.kqq, par, lim, p.status, abort_flag);
      ok0 = __all_sync(0xffffffffu, ok0);
      if (ok0) {
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue3<kDK / 8>(tmem + pr, tmem + T_S, tmem + T_LO, dkq_hi, dkq_lo, kq_step, id128, false);
          tc::mma_commit(&bars.pr);
        }
        __syncwarp();
        last = &bars.pr, last_par = par;
      }
    }
    // ---- meanwhile: F o K of this chunk (the previous update has read the
    // tile), then the next chunk's k and q in flight
    if (c > 0) {
      store_kt();
      publish(&bars.kt);
      write_out(c - 1);  // the previous chunk's O, in the other buffer
    }
    if (more) load_kq(c + 1);

    // ---- X = V - P' -> tf32 hi / lo; T' and B over the [E o K; E o Q] tile
    ok = ok0 && wait_or_abort(&bars.pr, par, lim, p.status, abort_flag);
    if (cta_any(!ok)) break;
    tc::fence_after_sync();
    if (vec) {  // v arrived as 16-byte pieces of four rows: to this thread's row
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float a[4] = {x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]};
        transpose4(a, lane);
        x[4 * i] = a[0], x[4 * i + 1] = a[1], x[4 * i + 2] = a[2], x[4 * i + 3] = a[3];
      }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // unrolled: x is indexed by q
      uint32_t w[16], hi[16], lo[16];
      tc::tmem_ld16(tl + pr + 32 * hf + 16 * q, w);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) tc::split_tf32(x[16 * q + e] - __uint_as_float(w[e]), hi[e], lo[e]);
      tc::tmem_st16(tl + T_LO + 32 * hf + 16 * q, hi);
      tc::tmem_st16(tl + T_LO + 64 + 32 * hf + 16 * q, lo);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int j4 = 16 * q4 + 4 * m;
      sts_split4(sm, OFF_THI + sq_off(trow, j4), OFF_TLO + sq_off(trow, j4), tv[m]);
      sts_split4(sm, OFF_BHI + sq_off(trow, j4), OFF_BLO + sq_off(trow, j4), bv[m]);
    }
    tc::tmem_wait_st();
    fence_proxy_async_smem();
    tc::fence_before_sync();
    mbar_arrive(&bars.xt);
    if (warp == 0 && ok0) {
      ok0 = __all_sync(0xffffffffu, wait_or_abort(&bars.xt, par, lim, p.status, abort_flag));
      if (ok0) {
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue3<kC / 8>(tmem + pr, tmem + T_LO, tmem + T_LO + 64, dt_hi, dt_lo, sq_step, id64, false);  // D
          tc::mma_commit(&bars.d);
        }
        __syncwarp();
        last = &bars.d, last_par = par;
      }
    }
    // ---- meanwhile: the next chunk's v, T', B and e_last in flight
    const float e_cur = e_last;
    if (more) load_rest(c + 1);

    // ---- S <- e_last S ([P' | R'], the last product reading S, is done)
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      uint32_t v[32];
      tc::tmem_ld32(tl + T_S + 64 * hf + 32 * q, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * e_cur);
      tc::tmem_st32(tl + T_S + 64 * hf + 32 * q, v);
    }

    // ---- D -> tf32 hi / lo (A of O and of the update)
    ok = ok0 && wait_or_abort(&bars.d, par, lim, p.status, abort_flag);
    if (cta_any(!ok)) break;
    tc::fence_after_sync();
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      uint32_t w[16], hi[16], lo[16];
      tc::tmem_ld16(tl + pr + 32 * hf + 16 * q, w);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) tc::split_tf32(__uint_as_float(w[e]), hi[e], lo[e]);
      tc::tmem_st16(tl + T_LO + 32 * hf + 16 * q, hi);
      tc::tmem_st16(tl + T_LO + 64 + 32 * hf + 16 * q, lo);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    mbar_arrive(&bars.dd);
    if (warp == 0 && ok0) {
      ok0 = wait_or_abort(&bars.dd, par, lim, p.status, abort_flag) &&
            wait_or_abort(&bars.kt, par, lim, p.status, abort_flag);
      ok0 = __all_sync(0xffffffffu, ok0);
      if (ok0) {
        tc::fence_after_sync();
        if (tc::elect_one()) {
          issue3<kC / 8>(tmem + pr + 64, tmem + T_LO, tmem + T_LO + 64, db_hi, db_lo, sq_step, id64, true);  // O
          tc::mma_commit(&bars.o);
          issue3<kC / 8>(tmem + T_S, tmem + T_LO, tmem + T_LO + 64, dkt_hi, dkt_lo, sq_step, id128, true);  // update
          tc::mma_commit(&bars.u);
        }
        __syncwarp();
        last = &bars.u, last_par = par;
      }
    }

    // ---- meanwhile: the next chunk's E o K over T' (D has read it)
    if (more) {
      store_rows(kr, 0);
      publish(&bars.kqk);
    }
    // ---- O done: the next chunk's E o Q over B, this chunk's outputs
    ok = ok0 && wait_or_abort(&bars.o, par, lim, p.status, abort_flag);
    if (cta_any(!ok)) break;
    tc::fence_after_sync();
    if (more) {
      store_rows(qr, kC);
      publish(&bars.kqq);
    }
    // ---- update done: lo of the next chunk's S
    ok = ok0 && wait_or_abort(&bars.u, par, lim, p.status, abort_flag);
    if (cta_any(!ok)) break;
    tc::fence_after_sync();
    if (more) split_state();
  }

  if (ok && nch > 0 && !*abort_flag) write_out(nch - 1);  // (uniform: ok and the flag are CTA-wide after the votes)

  // ---- final state -> the slot (every thread takes part in the vote)
  const bool fin = !cta_any(!ok || *abort_flag);
  if (fin) {
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
      uint32_t v[32];
      const int col0 = 64 * hf + 32 * q;
      tc::tmem_ld32(tl + T_S + col0, v);
      tc::tmem_wait_ld();
      if (row_ok) {
        if constexpr (sizeof(TS) == 4) {
          float4 *dst = reinterpret_cast<float4 *>(Sg + (int64_t)r * kDK + col0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                 __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(Sg + (int64_t)r * kDK + col0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t w4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[8 * e + 2 * k]),
                                                        __uint_as_float(v[8 * e + 2 * k + 1]));
              w4[k] = *reinterpret_cast<uint32_t *>(&b2);
            }
            dst[e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    }
  }
  // every MMA issued must be complete before the TMEM is freed
  if (tid == 0 && last) mbar_wait_bounded(last, last_par, p.drain_limit_ns);  // (warp 0 issued them)
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename TS>
int launch_chunked_tc_t(const RecurrentParams &p, cudaStream_t s) {
  static SmemLimit limit;  // per instantiation and device
  if (limit.ensure((const void *)chunked_tc_kernel<TS>, (int)kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  chunked_tc_kernel<TS><<<dim3(p.Hv, p.n_seq, 1), kThreads, kSmemBytes, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace

int launch_recurrent_chunked_tc(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (dk != kDK || p.dv > kMaxDv || p.dv < 1) return LSC_ERR_UNSUPPORTED;
  return ssm_dtype == LSC_BF16 ? launch_chunked_tc_t<__nv_bfloat16>(p, s) : launch_chunked_tc_t<float>(p, s);
}

}  // namespace lsc
