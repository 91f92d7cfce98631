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
// Per chunk and v head (M 128 = state rows, thread r = row r = TMEM lane r):
//   P'  = S (E o K)^T        N 64,  K 128   A = S from TMEM
//   R'  = S (E o Q)^T        N 64,  K 128   A = S from TMEM
//   D   = (V - P') T'^T      N 64,  K 64    A = X = V - P' from TMEM
//   O   = R' + D B^T         N 64,  K 64    A = D from TMEM  (o_t of every row)
//   S   = e_last S + D (F o K)   N 128, K 64    A = D from TMEM
// Products in tf32 with an fp32 accumulator.  Every operand x is split as
// x = hi + lo and each product formed as hi.hi + hi.lo + lo.hi: about 22
// significant bits per operand, so the products carry fp32-level error (the
// dropped lo.lo term is below 2^-21 of the product).  The tensor cores read a
// 32-bit operand as tf32 by truncation (its low 13 bits ignored), so the state
// in TMEM serves as its own hi part and only lo = tf32(S - trunc(S)) is
// written; the other operands use hi = tf32 rounded to nearest.
//
// CTA = one (sequence, v head), 256 threads, one CTA per SM (TMEM: all 512
// columns; shared memory ~201 KB):
//   warps 0-3   row warps: thread r owns state row r; thread 0 issues P', R',
//               D and O, thread 32 the state update (beside O), each once the
//               operands it reads are in place;
//   warps 4-7   producers: store the chunk's tf32 operand tiles into shared
//               memory as the products that read the previous contents finish
//               (E o K over the k half of the token-major tile, then T'; E o Q
//               over the q half, then B; channel-major F o K), loading k, q
//               and the records from global memory ahead of time.
// Hand-offs go through mbarriers: producers -> MMA (tiles in shared memory),
// row warps -> MMA (TMEM operands written, TMEM results read), MMA -> row
// warps / producers (tcgen05.commit).  Every wait is bounded: on expiry the
// thread records LSC_ERR_DEV_TIMEOUT, the CTA stops issuing work, waits
// (bounded) for the MMAs it issued and frees its TMEM.
//
// TMEM columns (lanes = state rows):
//   0-127    S (fp32; the hi part of its own split)
//   128-255  lo of S; after D: D hi (128-191), D lo (192-255)
//   256-319  P'; after X is formed: D
//   320-447  X hi (320-383), X lo (384-447)
//   448-511  R', then O = R' + D B^T
// Shared-memory tiles (no swizzle, lsc_chunk.h): the token-major [E o K; E o Q]
// tile (hi, lo), T' over its k half once P' has read it, B over its q half
// once R' has; F o K channel-major (hi, lo).
#include "lsc_chunk.h"
#include "lsc_gdn_common.cuh"
#include "lsc_tc.h"

namespace lsc {
namespace {

using namespace chunk;

constexpr int kThreads = 256;
constexpr int kRowThreads = 128;
constexpr int kProd0 = 128;  // first producer thread
constexpr uint32_t kTmemCols = 512;

constexpr uint32_t T_S = 0;
constexpr uint32_t T_SLO = 128;
constexpr uint32_t T_DHI = 128, T_DLO = 192;
constexpr uint32_t T_P = 256, T_D = 256;
constexpr uint32_t T_XHI = 320, T_XLO = 384;
constexpr uint32_t T_R = 448;

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

// Row warps (warps 0-3) synchronise among themselves on named barrier 1, in
// the non-aligned forms (thread 0 may arrive apart from its warp), and leave
// with the warp reconverged for the warp-wide .sync.aligned TMEM loads and
// stores that follow.
__device__ __forceinline__ void named_sync_rows() {
  asm volatile("barrier.sync 1, 128;" ::: "memory");
  __syncwarp();
}
// true on every row thread when v is true on any of them
__device__ __forceinline__ bool named_any_rows(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "barrier.red.or.pred p, 1, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  __syncwarp();
  return r != 0;
}

struct Bars {
  uint64_t kqk, kqq, tk, tq, kt;  // producers: E o K, E o Q, T', B, F o K stored
  uint64_t split, xt, dd;         // row warps: lo of S, X, D hi / lo (and the decayed S) written
  uint64_t p, r, d, o, u;         // MMA commits
};

// 64 TMEM columns of this thread's lane as floats, one wait
__device__ __forceinline__ void ld64(uint32_t taddr, float (&x)[kC]) {
  uint32_t a[16], b[16], c[16], d[16];
  tc::tmem_ld16(taddr, a);
  tc::tmem_ld16(taddr + 16, b);
  tc::tmem_ld16(taddr + 32, c);
  tc::tmem_ld16(taddr + 48, d);
  tc::tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    x[e] = __uint_as_float(a[e]);
    x[16 + e] = __uint_as_float(b[e]);
    x[32 + e] = __uint_as_float(c[e]);
    x[48 + e] = __uint_as_float(d[e]);
  }
}

__device__ __forceinline__ void sts_split4(uint8_t *sm, uint32_t off_hi, uint32_t off_lo, float4 f) {
  uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
  tc::split_tf32(f.x, h0, l0);
  tc::split_tf32(f.y, h1, l1);
  tc::split_tf32(f.z, h2, l2);
  tc::split_tf32(f.w, h3, l3);
  *reinterpret_cast<uint4 *>(sm + off_hi) = make_uint4(h0, h1, h2, h3);
  *reinterpret_cast<uint4 *>(sm + off_lo) = make_uint4(l0, l1, l2, l3);
}

__device__ __forceinline__ float4 scale4(float4 v, float s) { return make_float4(v.x * s, v.y * s, v.z * s, v.w * s); }

// lo part of x when the tensor cores read x itself as its hi part (truncation)
__device__ __forceinline__ uint32_t lo_of_truncated(float x) {
  return tc::to_tf32(x - __uint_as_float(__float_as_uint(x) & 0xffffe000u));
}

// ---- MMA issue (one thread; three tf32 passes per product, unrolled) --------
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
    mbar_init(&bars.kqk, kThreads - kProd0);  // every producer thread
    mbar_init(&bars.kqq, kThreads - kProd0);
    mbar_init(&bars.tk, kThreads - kProd0);
    mbar_init(&bars.tq, kThreads - kProd0);
    mbar_init(&bars.kt, kThreads - kProd0);
    mbar_init(&bars.split, kRowThreads);
    mbar_init(&bars.xt, kRowThreads);
    mbar_init(&bars.dd, kRowThreads);
    mbar_init(&bars.p, 1);
    mbar_init(&bars.r, 1);
    mbar_init(&bars.d, 1);
    mbar_init(&bars.o, 1);
    mbar_init(&bars.u, 1);
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

  if (warp < 4) {
    // ======================================================= row warps
    const int r = tid;
    const bool row_ok = r < dv;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes
    constexpr uint32_t id64 = tc::idesc_tf32(128, 64, false);
    constexpr uint32_t id128 = tc::idesc_tf32(128, 128, false);
    // B operand descriptors; a k step of 8 tf32 columns is 256 bytes along
    // the token-major tile, 2 kLbo bytes along a 64-column tile
    const uint64_t dk_hi = tc::smem_desc(smem_u32(sm + OFF_KQHI), 128, kKqRg);
    const uint64_t dk_lo = tc::smem_desc(smem_u32(sm + OFF_KQLO), 128, kKqRg);
    const uint64_t dq_hi = tc::smem_desc(smem_u32(sm + OFF_KQHI + kQRow0), 128, kKqRg);
    const uint64_t dq_lo = tc::smem_desc(smem_u32(sm + OFF_KQLO + kQRow0), 128, kKqRg);
    const uint64_t dt_hi = tc::smem_desc(smem_u32(sm + OFF_THI), kLbo, kRg64);
    const uint64_t dt_lo = tc::smem_desc(smem_u32(sm + OFF_TLO), kLbo, kRg64);
    const uint64_t db_hi = tc::smem_desc(smem_u32(sm + OFF_BHI), kLbo, kRg64);
    const uint64_t db_lo = tc::smem_desc(smem_u32(sm + OFF_BLO), kLbo, kRg64);
    const uint64_t dkt_hi = tc::smem_desc(smem_u32(sm + OFF_KTHI), kLbo, kRg64);
    const uint64_t dkt_lo = tc::smem_desc(smem_u32(sm + OFF_KTLO), kLbo, kRg64);
    constexpr uint32_t kq_step = 256 >> 4, sq_step = (2 * kLbo) >> 4;
    uint64_t *last = nullptr;  // the last commit's barrier and phase (threads 0 and 32)
    uint32_t last_par = 0;
    auto commit = [&](uint64_t *bar, uint32_t par) {
      tc::mma_commit(bar);
      last = bar, last_par = par;
    };
    // initial state -> TMEM (zero when cold; rows >= dv stay zero)
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = 0u;
      if (warm && row_ok) {
        if constexpr (sizeof(TS) == 4) {
          const float4 *src = reinterpret_cast<const float4 *>(Sg + (int64_t)r * kDK + 32 * q);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 f = __ldg(src + e);
            v[4 * e] = __float_as_uint(f.x);
            v[4 * e + 1] = __float_as_uint(f.y);
            v[4 * e + 2] = __float_as_uint(f.z);
            v[4 * e + 3] = __float_as_uint(f.w);
          }
        } else {
          const uint4 *src = reinterpret_cast<const uint4 *>(Sg + (int64_t)r * kDK + 32 * q);
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
      tc::tmem_st32(tl + T_S + 32 * q, v);
    }
    tc::tmem_wait_st();

#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
      const uint32_t par = c & 1;
      const int nt = min(kC, t1 - t0 - c * kC);
      const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
      const float *rec = recs + c * rec_stride;
      // v_t[r] of this chunk, in flight during the first steps
      float x[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t)
        x[t] = (t < nt && row_ok) ? __ldg(p.v + ((tb + t) * p.Hv + h) * dv + r) : 0.f;
      const float e_last = __ldg(rec + kRecMisc);

      // ---- 1: lo of S (the update of the previous chunk is complete)
      bool ok0 = true;
      bool ok = c == 0 || wait_or_abort(&bars.u, par ^ 1, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
#pragma unroll 1
      for (int q = 0; q < kDK / 32; ++q) {
        uint32_t v[32];
        tc::tmem_ld32(tl + T_S + 32 * q, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = lo_of_truncated(__uint_as_float(v[e]));
        tc::tmem_st32(tl + T_SLO + 32 * q, v);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars.split);
      if (r == 0) {
        if ((ok0 = wait_or_abort(&bars.split, par, lim, p.status, abort_flag) &&
                   wait_or_abort(&bars.kqk, par, lim, p.status, abort_flag))) {
          tc::fence_after_sync();
          issue3<kDK / 8>(tmem + T_P, tmem + T_S, tmem + T_SLO, dk_hi, dk_lo, kq_step, id64, false);  // P'
          commit(&bars.p, par);
        }
        if (ok0 && (ok0 = wait_or_abort(&bars.kqq, par, lim, p.status, abort_flag))) {
          tc::fence_after_sync();
          issue3<kDK / 8>(tmem + T_R, tmem + T_S, tmem + T_SLO, dq_hi, dq_lo, kq_step, id64, false);  // R'
          commit(&bars.r, par);
        }
      }
      __syncwarp();

      // ---- 2: X = V - P' -> tf32 hi / lo
      ok = ok0 && wait_or_abort(&bars.p, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      {
        float pv[kC];
        ld64(tl + T_P, pv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) tc::split_tf32(x[16 * q + e] - pv[16 * q + e], hi[e], lo[e]);
          tc::tmem_st16(tl + T_XHI + 16 * q, hi);
          tc::tmem_st16(tl + T_XLO + 16 * q, lo);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars.xt);
      if (r == 0 && ok0 &&
          (ok0 = wait_or_abort(&bars.xt, par, lim, p.status, abort_flag) &&
                 wait_or_abort(&bars.tk, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue3<kC / 8>(tmem + T_D, tmem + T_XHI, tmem + T_XLO, dt_hi, dt_lo, sq_step, id64, false);  // D
        commit(&bars.d, par);
      }
      __syncwarp();

      // ---- 3: S <- e_last S once R' (the last product reading S) is done
      ok = ok0 && wait_or_abort(&bars.r, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
#pragma unroll 1
      for (int q = 0; q < kDK / 32; ++q) {
        uint32_t v[32];
        tc::tmem_ld32(tl + T_S + 32 * q, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * e_last);
        tc::tmem_st32(tl + T_S + 32 * q, v);
      }

      // ---- 4: D -> tf32 hi / lo (A of O and of the update)
      ok = ok0 && wait_or_abort(&bars.d, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      {
        float dvv[kC];
        ld64(tl + T_D, dvv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) tc::split_tf32(dvv[16 * q + e], hi[e], lo[e]);
          tc::tmem_st16(tl + T_DHI + 16 * q, hi);
          tc::tmem_st16(tl + T_DLO + 16 * q, lo);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars.dd);
      // O (thread 0) and the update (thread 32) read the same A operand: two
      // issuing threads keep the tensor core fed
      if (r == 0 && ok0 &&
          (ok0 = wait_or_abort(&bars.dd, par, lim, p.status, abort_flag) &&
                 wait_or_abort(&bars.tq, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue3<kC / 8>(tmem + T_R, tmem + T_DHI, tmem + T_DLO, db_hi, db_lo, sq_step, id64, true);  // O
        commit(&bars.o, par);
      } else if (r == 32 && (ok0 = wait_or_abort(&bars.dd, par, lim, p.status, abort_flag) &&
                                   wait_or_abort(&bars.kt, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue3<kC / 8>(tmem + T_S, tmem + T_DHI, tmem + T_DLO, dkt_hi, dkt_lo, sq_step, id128, true);  // update
        commit(&bars.u, par);
      }
      __syncwarp();

      // ---- 5: outputs
      ok = ok0 && wait_or_abort(&bars.o, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      {
        float *o = p.out + (tb * p.Hv + h) * dv + r;
        const int64_t ostride = (int64_t)p.Hv * dv;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t w[16];
          tc::tmem_ld16(tl + T_R + 16 * q, w);
          tc::tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (16 * q + e < nt) o[(16 * q + e) * ostride] = __uint_as_float(w[e]);
          }
        }
      }
      tc::fence_before_sync();
      named_sync_rows();  // every row has read O: the next R' may overwrite it
    }
    // ---- final state -> the slot
    const bool fin = nch == 0 || wait_or_abort(&bars.u, (nch - 1) & 1, lim, p.status, abort_flag);
    if (!named_any_rows(!fin || *abort_flag)) {
      tc::fence_after_sync();
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        __syncwarp();
        tc::tmem_ld32(tl + T_S + 32 * q, v);
        tc::tmem_wait_ld();
        if (row_ok) {
          if constexpr (sizeof(TS) == 4) {
            float4 *dst = reinterpret_cast<float4 *>(Sg + (int64_t)r * kDK + 32 * q);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>(Sg + (int64_t)r * kDK + 32 * q);
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
    // every MMA issued must be complete before the TMEM is freed (threads 0
    // and 32 each wait for their own last commit)
    if ((r == 0 || r == 32) && last) mbar_wait_bounded(last, last_par, p.drain_limit_ns);
    tc::fence_before_sync();
  } else {
    // ======================================================= producers
    const int pt = tid - kProd0, pw = pt >> 5;
    const int al = lane & 7, bl = lane >> 3;
    // k and q of a chunk: [token block half][channel block half][token in
    // block]; this thread's 4 x 4 blocks are tokens 4a..4a+3, channels
    // 4b..4b+3 with a = al + 8 ah, b = bl + 4 pw + 16 bh; E and F of its tokens
    float4 kr[2][2][4], qr[2][2][4];
    float ev[2][4], fv[2][4];
    auto load_kq = [&](int c) {
      const int nt = min(kC, t1 - t0 - c * kC);
      const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
      const float *rec = recs + c * rec_stride;
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = 4 * (al + 8 * ah) + u;
          ev[ah][u] = __ldg(rec + kRecE + tok);
          fv[ah][u] = __ldg(rec + kRecF + tok);
#pragma unroll
          for (int bh = 0; bh < 2; ++bh) {
            const int b = bl + 4 * pw + 16 * bh;
            const int64_t off = ((tb + tok) * p.Hk + g) * kDK + 4 * b;
            const bool in = tok < nt;
            kr[ah][bh][u] = in ? __ldg(reinterpret_cast<const float4 *>(p.k + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
            qr[ah][bh][u] = in ? __ldg(reinterpret_cast<const float4 *>(p.q + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
    };
    // token-major E o K (rows 0-63) or E o Q (rows 64-127)
    auto store_rows = [&](const float4 (&src)[2][2][4], int row0) {
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int bh = 0; bh < 2; ++bh)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * (al + 8 * ah) + u, c4 = 4 * (bl + 4 * pw + 16 * bh);
            sts_split4(sm, OFF_KQHI + kq_off(row0 + j, c4), OFF_KQLO + kq_off(row0 + j, c4),
                       scale4(src[ah][bh][u], ev[ah][u]));
          }
    };
    // channel-major F o K: K[j][c] F_j at (channel c, token j)
    auto store_kt = [&]() {
#pragma unroll
      for (int ah = 0; ah < 2; ++ah) {
        const int a = al + 8 * ah;
        const float f0 = fv[ah][0], f1 = fv[ah][1], f2 = fv[ah][2], f3 = fv[ah][3];
#pragma unroll
        for (int bh = 0; bh < 2; ++bh) {
          const int b = bl + 4 * pw + 16 * bh;
          const float4 *k4 = kr[ah][bh];
          const float col[4][4] = {{k4[0].x * f0, k4[1].x * f1, k4[2].x * f2, k4[3].x * f3},
                                   {k4[0].y * f0, k4[1].y * f1, k4[2].y * f2, k4[3].y * f3},
                                   {k4[0].z * f0, k4[1].z * f1, k4[2].z * f2, k4[3].z * f3},
                                   {k4[0].w * f0, k4[1].w * f1, k4[2].w * f2, k4[3].w * f3}};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ch = 4 * b + e;
            sts_split4(sm, OFF_KTHI + sq_off(ch, 4 * a), OFF_KTLO + sq_off(ch, 4 * a),
                       make_float4(col[e][0], col[e][1], col[e][2], col[e][3]));
          }
        }
      }
    };
    // T' and B of a chunk: row pt / 2, columns 32 (pt % 2) .. + 31 (the
    // 16-byte groups past the diagonal's are zero and not read)
    const int trow = pt >> 1, tj0 = 32 * (pt & 1);
    float4 tv[8], bv[8];
    auto load_tb = [&](int c) {
      const float *rec = recs + c * rec_stride;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int j4 = tj0 + 4 * m;
        const bool in = j4 < 4 * row_groups(trow);
        tv[m] = in ? __ldg(reinterpret_cast<const float4 *>(rec + kRecT + trow * kC + j4)) : make_float4(0.f, 0.f, 0.f, 0.f);
        bv[m] = in ? __ldg(reinterpret_cast<const float4 *>(rec + kRecB + trow * kC + j4)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    auto store_sq = [&](const float4 (&src)[8], uint32_t off_hi, uint32_t off_lo) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        sts_split4(sm, off_hi + sq_off(trow, tj0 + 4 * m), off_lo + sq_off(trow, tj0 + 4 * m), src[m]);
    };
    auto publish = [&](uint64_t *bar) {
      fence_proxy_async_smem();  // generic-proxy stores, read by the MMA
      mbar_arrive(bar);
    };

    // Chunk c's tiles are stored as the products reading the previous
    // contents finish: T' after P'(c), B after R'(c); then the next chunk's
    // E o K after D(c), E o Q after O(c), F o K after the update of chunk c.
    if (nch > 0) {
      load_kq(0);
      store_rows(kr, 0);
      publish(&bars.kqk);
      store_rows(qr, kC);
      publish(&bars.kqq);
      store_kt();
      publish(&bars.kt);
      load_tb(0);
    }
#pragma unroll 1
    for (int c = 0; c < nch && !*abort_flag; ++c) {
      const uint32_t par = c & 1;
      if (!wait_or_abort(&bars.p, par, lim, p.status, abort_flag)) break;
      store_sq(tv, OFF_THI, OFF_TLO);
      publish(&bars.tk);
      if (!wait_or_abort(&bars.r, par, lim, p.status, abort_flag)) break;
      store_sq(bv, OFF_BHI, OFF_BLO);
      publish(&bars.tq);
      if (c + 1 == nch) break;
      load_kq(c + 1);
      if (!wait_or_abort(&bars.d, par, lim, p.status, abort_flag)) break;
      store_rows(kr, 0);
      publish(&bars.kqk);
      if (!wait_or_abort(&bars.o, par, lim, p.status, abort_flag)) break;
      store_rows(qr, kC);
      publish(&bars.kqq);
      if (!wait_or_abort(&bars.u, par, lim, p.status, abort_flag)) break;
      store_kt();
      publish(&bars.kt);
      load_tb(c + 1);
    }
  }

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
