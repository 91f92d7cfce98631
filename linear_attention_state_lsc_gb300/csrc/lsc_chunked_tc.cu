// lsc_chunked_tc.cu -- the resumed-prefill GDN recurrence evaluated 64 tokens
// at a time on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
// Same token-ordered result as the token-by-token kernels (per token
// S' = a S (I - b k k^T) + b v k^T, o = S' q), rearranged so that the work of
// a chunk is a handful of matrix products plus a small triangular inverse.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule, the token recurrence)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with
//        q); "相同前缀不一定能全部复用" (continue from the restored checkpoint)
// The pages give the token recurrence only; the chunked form is its algebraic
// rearrangement, exact up to rounding.
//
// One chunk, tokens 0..C-1, from state S (dv x dk, rows r):
//   Gam(j,t) = a_(j+1) ... a_t,  E_t = a_0 ... a_t,  F_j = Gam(j, C-1)
//   P = S K^T, R = S Q^T (dv x C),  G_jt = k_j.k_t,  M_jt = k_j.q_t
//   A_tj = b_t Gam(j,t) G_jt (j < t),  T = (I + A)^-1 (unit lower triangular)
//   X_rt = b_t (v_t[r] - E_t P_rt),  D = X T^T    (d_t = x_t - sum_(j<t) A_tj d_j)
//   B_tj = Gam(j,t) M_jt (j <= t),   O = E o R + D B^T   (o_t of every row)
//   S' = E_(C-1) S + D (F o K)                     (the rank-C update)
// Gam is formed from a per-chunk running sum of log2|a| (zeros and signs of a
// tracked apart), so no product of gates under- or overflows on the way.
//
// Products on the tensor cores, in tf32 with an fp32 accumulator.  Every
// operand x is split as x = hi + lo (hi = tf32(x), lo = tf32(x - hi)) and each
// product is formed as hi.hi + hi.lo + lo.hi: about 22 significant bits per
// operand, so the products carry fp32-level error (the dropped lo.lo term is
// below 2^-21 of the product).  Per chunk and v head (M 128 = state rows):
//   Gram    [K;Q] K^T           M 128 (k rows, q rows), N 64,  K 128 (smem)
//   P | R   S [K;Q]^T           N 128, K 128   A = S from TMEM
//   D       X T^T               N 64,  K 64    A = X from TMEM
//   O       E o R + D B^T       N 64,  K 64    A = D from TMEM
//   update  S += D (F o K)      N 128, K 64    A = D from TMEM
// The state lives in TMEM as the update's accumulator and is decayed by
// E_(C-1) in place each chunk.  The CUDA cores form A and B from the Gram
// accumulator (one row per thread), invert I + A by 16 x 16 blocks (the
// diagonal blocks by forward substitution, then three levels of block
// products), and split the TMEM operands; one thread per state row.
//
// CTA = one (sequence, v head), 256 threads, one CTA per SM (TMEM: all 512
// columns; shared memory: ~224 KB):
//   warps 0-3   row warps: thread r owns state row r (TMEM lane r) and row r
//               of A (r < 64) or of B (r >= 64); warp 0 allocates the TMEM
//               and thread 0 issues the MMAs and commits once the operands
//               they read are in place, thread 32 the state update beside
//               thread 0's O product (two warps per SM sub-partition leave
//               each thread up to 255 registers);
//   warps 4-7   producers: load the next chunk's k and q from global memory
//               into registers while the current chunk runs, split them and
//               store them as tf32 operands (token-major [K; Q] once the
//               current chunk's products that overlay that tile are done,
//               channel-major F o K once its update is done), and form the
//               next chunk's gate scan.
// Hand-offs go through mbarriers: producer -> MMA (operands in shared
// memory), row warps -> MMA (TMEM operands written, TMEM results read), MMA
// -> row warps / producers (tcgen05.commit).  Every wait is bounded: on
// expiry the thread records LSC_ERR_DEV_TIMEOUT, the CTA stops issuing work,
// waits (bounded) for the MMAs it issued and frees its TMEM.  The per-chunk
// code runs as rolled loops with small bodies: each chunk executes it once,
// and straight-line code of that size would be fetched from L2 every chunk.
//
// Shared-memory operands (no swizzle, 8 x 16-byte core matrices):
//   [K; Q] token-major: element (row i, channel c) at (i/8)*4112 + (c/4)*128 +
//   (i%8)*16 + (c%4)*4 -- K-major with LBO 128, SBO 4112 (rows 0-63 k, 64-127 q);
//   F o K channel-major: element (channel c, token j) at (c/8)*2304 +
//   (j/4)*144 + (c%8)*16 + (j%4)*4 -- K-major with LBO 144, SBO 2304;
//   T and B (64 x 64, row t, column j) at (t/8)*2304 + (j/4)*144 + (t%8)*16 +
//   (j%4)*4: T over the k rows and B over the q rows of the [K; Q] tiles once
//   P | R has read them.
// The 16 bytes beyond each 4096 (resp. 128) spread the threads' stores over
// all banks.
#include "lsc_gdn_common.cuh"
#include "lsc_tc.h"

namespace lsc {
namespace {

constexpr int kC = 64;        // tokens per chunk
constexpr int kDK = 128;      // head_k_dim of this kernel
constexpr int kThreads = 256;
constexpr int kRowThreads = 128;
constexpr int kProd0 = 128;   // first producer thread
constexpr uint32_t kTmemCols = 512;

// TMEM columns (lane = state row for every accumulator and A operand)
constexpr uint32_t T_S = 0;      // state, fp32 (128)
constexpr uint32_t T_SHI = 128;  // tf32 hi of S (128)      -> X hi (64), X lo (64)
constexpr uint32_t T_SLO = 256;  // tf32 lo of S (128)      -> D (64), D hi (64)
constexpr uint32_t T_P = 384;    // P (64)                  -> x, then D lo (64)
constexpr uint32_t T_R = 448;    // Gram (64), then R -> E o R -> O (64)
constexpr uint32_t T_XHI = 128, T_XLO = 192;
constexpr uint32_t T_D = 256, T_DHI = 320, T_DLO = 384;

// shared-memory layout (bytes)
constexpr uint32_t kKqRg = 4096 + 16;      // one 8-row group of the token-major tile
constexpr uint32_t kKqBytes = 16 * kKqRg;  // 128 rows
constexpr uint32_t kQRow0 = 8 * kKqRg;     // q rows start at row 64
constexpr uint32_t kLbo = 128 + 16;        // one 4-column core-matrix column of a 64-column tile
constexpr uint32_t kRg64 = 16 * kLbo;      // one 8-row group of a 64-column tile
constexpr uint32_t kKtBytes = 16 * kRg64;  // channel-major K: 128 channel rows
constexpr uint32_t kSqBytes = 8 * kRg64;   // T or B: 64 rows

// Packed triangles (fp32), every row a multiple of 4 floats, 16-byte aligned:
// A by rows (row t: columns j in [0, 4 ceil(t/4)), zero for j >= t), T by
// rows including the diagonal (row t: columns j in [0, 4 floor(t/4) + 4),
// zero for j > t).
__host__ __device__ constexpr int a1_of(int t) { return 4 * ((t + 3) / 4); }
__host__ __device__ constexpr int b1_of(int t) { return 4 * ((t + 4) / 4); }
// sum over m = 1..n of floor(m / 4)
__host__ __device__ constexpr int quarter_sum(int n) {
  return n <= 0 ? 0 : 2 * (n / 4) * (n / 4 - 1) + (n / 4) * (n % 4 + 1);
}
__host__ __device__ constexpr int a_row(int t) { return 4 * quarter_sum(t + 2); }      // sum of a1_of(i), i < t
__host__ __device__ constexpr int t_row(int t) { return 4 * t + 4 * quarter_sum(t - 1); }  // sum of b1_of(i), i < t
static_assert(a_row(1) == 0 && a_row(2) == 4 && a_row(5) == 16 && t_row(1) == 4 && t_row(5) == 4 * 4 + 8, "packing");
constexpr int kAFloats = a_row(kC);
constexpr int kTFloats = t_row(kC);
constexpr int kYFloats = 3 * 16 * 16;  // block-product scratch of the inverse

// per-chunk gate quantities, formed by the producers (double-buffered)
struct ChunkGates {
  float beta[kC];
  float cum[kC];   // running sum of log2|a_t| over the chunk (0 where a_t = 0)
  float E[kC];     // a_0 ... a_t
  float F[kC];     // Gam(t, C-1)
  int32_t seg[kC];   // last t' <= t with a_t' = 0, or -1
  int32_t nneg[kC];  // number of negative a_t' for t' <= t
  float e_last;
  int32_t pad[3];
};

constexpr uint32_t OFF_KQHI = 0;
constexpr uint32_t OFF_KQLO = OFF_KQHI + kKqBytes;
constexpr uint32_t OFF_KTHI = OFF_KQLO + kKqBytes;
constexpr uint32_t OFF_KTLO = OFF_KTHI + kKtBytes;
constexpr uint32_t OFF_A = OFF_KTLO + kKtBytes;
constexpr uint32_t OFF_TP = OFF_A + 4 * kAFloats;
constexpr uint32_t OFF_Y = OFF_TP + 4 * kTFloats;
constexpr uint32_t OFF_GATES = OFF_Y + 4 * kYFloats;
constexpr uint32_t kSmemBytes = OFF_GATES + 2 * sizeof(ChunkGates);
// T and B operands (hi, lo) over the [K; Q] tiles, written once P | R is done
constexpr uint32_t OFF_THI = OFF_KQHI, OFF_TLO = OFF_KQLO;
constexpr uint32_t OFF_BHI = OFF_KQHI + kQRow0, OFF_BLO = OFF_KQLO + kQRow0;
static_assert(kSqBytes <= kQRow0 && kQRow0 + kSqBytes <= kKqBytes, "T over the k rows, B over the q rows");
static_assert(OFF_A % 16 == 0 && OFF_TP % 16 == 0 && OFF_Y % 16 == 0 && OFF_GATES % 16 == 0, "alignment");
static_assert(kSmemBytes <= 226 * 1024, "shared memory budget (one CTA per SM)");

// byte offset of (row, col) in a 64-column operand tile
__host__ __device__ constexpr uint32_t sq_off(int row, int col) {
  return (uint32_t)(row / 8) * kRg64 + (uint32_t)(col / 4) * kLbo + (uint32_t)(row % 8) * 16 + (uint32_t)(col % 4) * 4;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));  // results below 2^-126 flush to 0
  return y;
}

// Gam(j, t) for j <= t (j = -1: E_t)
__device__ __forceinline__ float gam(const ChunkGates &G, int j, int t) {
  if (G.seg[t] > j) return 0.f;
  const float c0 = j >= 0 ? G.cum[j] : 0.f;
  const int n0 = j >= 0 ? G.nneg[j] : 0;
  const float m = ex2(G.cum[t] - c0);
  return ((G.nneg[t] - n0) & 1) ? -m : m;
}

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
  uint64_t kq, kt, gates, split, ab, xt, dd;  // arrivals
  uint64_t g, pr, d, o, u;                    // MMA commits
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

// T = (I + A)^-1 by 16 x 16 blocks, on the 128 row threads (rows and the
// diagonal of T packed by rows at Tp; A packed by rows at Ap; Y is scratch).
//   diagonal blocks:  T_bb = (I + A_bb)^-1 by forward substitution, thread
//                     16 b + jj forming column jj of T_bb;
//   level L = 1..3:   Y_ab = sum_(b<=m<a) A_am T_mb, then T_ab = -T_aa Y_ab,
//                     for a = b + L; one work item = (block, row, 4 columns).
// Row offsets inside a 16-row block: the rows 16 m + i of a packed triangle
// start at row(16 m) + 16 m i + row(i) (each row of the block is 16 m longer
// than row i of the first block), so only row(16 m) is formed at run time.
__device__ __forceinline__ float4 mask_above(float4 v, int col0, int row) {  // zero the entries with col > row
  if (col0 > row) v.x = 0.f;
  if (col0 + 1 > row) v.y = 0.f;
  if (col0 + 2 > row) v.z = 0.f;
  if (col0 + 3 > row) v.w = 0.f;
  return v;
}
__device__ __forceinline__ void fma4(float4 &acc, float s, const float4 &v) {
  acc.x = fmaf(s, v.x, acc.x);
  acc.y = fmaf(s, v.y, acc.y);
  acc.z = fmaf(s, v.z, acc.z);
  acc.w = fmaf(s, v.w, acc.w);
}
__device__ __forceinline__ void invert_unit_lower(const float *Ap, float *Tp, float *Y, int r) {
  if (r < kC) {
    const int b = r / 16, jj = r % 16, b16 = 16 * b;
    const float *ab = Ap + a_row(b16) + b16;  // + 16 b tt + a_row(tt) + n gives A(16 b + tt, 16 b + n)
    float acc[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) acc[tt] = tt == jj ? 1.f : 0.f;
#pragma unroll
    for (int n = 0; n < 15; ++n) {
      const float tn = acc[n];
#pragma unroll
      for (int tt = n + 1; tt < 16; ++tt) acc[tt] = fmaf(-ab[b16 * tt + a_row(tt) + n], tn, acc[tt]);
    }
    float *tb = Tp + t_row(b16) + b16 + jj;  // + 16 b tt + t_row(tt) gives T(16 b + tt, 16 b + jj)
#pragma unroll
    for (int tt = 0; tt < 16; ++tt)
      if (tt >= jj) tb[b16 * tt + t_row(tt)] = acc[tt];
  }
  named_sync_rows();
  float4 *Y4 = reinterpret_cast<float4 *>(Y);
#pragma unroll 1
  for (int L = 1; L < 4; ++L) {
    const int nitems = (4 - L) * 64;
    // Y_ab(i, 4 q .. 4 q + 3) = sum over m in [b, a) and kk of A(16 a + i, 16 m + kk) T(16 m + kk, 16 b + 4 q ..)
#pragma unroll 1
    for (int e = r; e < nitems; e += kRowThreads) {
      const int bb = e / 64, i = (e / 4) % 16, q = e % 4, a = bb + L, col = 16 * bb + 4 * q;
      const float *arow = Ap + a_row(16 * a + i);
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
      for (int m = bb; m < a; ++m) {
        const int m16 = 16 * m;
        const float *tm = Tp + t_row(m16) + col;  // + 16 m kk + t_row(kk) gives T(16 m + kk, col)
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const float4 av = *reinterpret_cast<const float4 *>(arow + m16 + 4 * k4);
          const float as[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const int kk = 4 * k4 + e2;
            const float4 tv = mask_above(*reinterpret_cast<const float4 *>(tm + m16 * kk + t_row(kk)), col, m16 + kk);
            fma4(y, as[e2], tv);
          }
        }
      }
      Y4[e] = y;  // [block][row i][4-column group q]
    }
    named_sync_rows();
    // T_ab(i, 4 q ..) = -sum over kk <= i of T(16 a + i, 16 a + kk) Y_ab(kk, 4 q ..)
#pragma unroll 1
    for (int e = r; e < nitems; e += kRowThreads) {
      const int bb = e / 64, i = (e / 4) % 16, q = e % 4, a = bb + L;
      float *trow = Tp + t_row(16 * a + i);
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const float4 tv = mask_above(*reinterpret_cast<const float4 *>(trow + 16 * a + 4 * k4), 4 * k4, i);
        const float ts[4] = {tv.x, tv.y, tv.z, tv.w};
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) fma4(t, ts[e2], Y4[bb * 64 + (4 * k4 + e2) * 4 + q]);
      }
      *reinterpret_cast<float4 *>(trow + 16 * bb + 4 * q) = make_float4(-t.x, -t.y, -t.z, -t.w);
    }
    named_sync_rows();
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
  ChunkGates *gates = reinterpret_cast<ChunkGates *>(sm + OFF_GATES);
  TS *Sg = reinterpret_cast<TS *>(p.layer + (int64_t)slot * p.page + p.ssm_off) + (int64_t)h * dv * kDK;

  if (tid == 0) {
    mbar_init(&bars.kq, kThreads - kProd0);  // every producer thread
    mbar_init(&bars.kt, kThreads - kProd0);
    mbar_init(&bars.gates, 1);
    mbar_init(&bars.split, kRowThreads);
    mbar_init(&bars.ab, kRowThreads);
    mbar_init(&bars.xt, kRowThreads);
    mbar_init(&bars.dd, kRowThreads);
    mbar_init(&bars.g, 1);
    mbar_init(&bars.pr, 1);
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
    // MMA issue (thread 0): three tf32 passes (hi.hi, hi.lo, lo.hi) per
    // product.  The issue loops stay rolled and advance the descriptors by
    // constants (the start address sits in the descriptor's low bits): a k
    // step of 8 tf32 columns is 256 bytes along a 128-column tile, 288 bytes
    // along a 64-column tile, 8 columns of a TMEM operand.
    const uint32_t kqhi = smem_u32(sm + OFF_KQHI), kqlo = smem_u32(sm + OFF_KQLO);
    const uint32_t kthi = smem_u32(sm + OFF_KTHI), ktlo = smem_u32(sm + OFF_KTLO);
    const uint32_t thi = smem_u32(sm + OFF_THI), tlo = smem_u32(sm + OFF_TLO);
    const uint32_t bhi = smem_u32(sm + OFF_BHI), blo = smem_u32(sm + OFF_BLO);
    constexpr uint32_t id64 = tc::idesc_tf32(128, 64, false);
    constexpr uint32_t id128 = tc::idesc_tf32(128, 128, false);
    uint64_t *last = nullptr;  // the last commit's barrier and phase (threads 0 and 32)
    uint32_t last_par = 0;
    auto commit = [&](uint64_t *bar, uint32_t par) {
      tc::mma_commit(bar);
      last = bar, last_par = par;
    };
    // [K;Q] (128 rows) x K (64 rows)^T -> T_R
    auto issue_gram = [&]() {
#pragma unroll 1
      for (int ps = 0; ps < 3; ++ps) {
        uint64_t ad = tc::smem_desc(ps == 2 ? kqlo : kqhi, 128, kKqRg);
        uint64_t bd = tc::smem_desc(ps == 1 ? kqlo : kqhi, 128, kKqRg);
#pragma unroll 1
        for (int s = 0; s < kDK / 8; s += 4, ad += 4 * (256 >> 4), bd += 4 * (256 >> 4)) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            tc::mma_ss(tmem + T_R, ad + u * (256 >> 4), bd + u * (256 >> 4), id64, (ps | s | u) != 0);
        }
      }
    };
    // S x [K;Q]^T -> T_P (P) | T_R (R)
    auto issue_pr = [&]() {
#pragma unroll 1
      for (int ps = 0; ps < 3; ++ps) {
        uint32_t a = tmem + (ps == 2 ? T_SLO : T_SHI);
        uint64_t bd = tc::smem_desc(ps == 1 ? kqlo : kqhi, 128, kKqRg);
#pragma unroll 1
        for (int s = 0; s < kDK / 8; s += 4, a += 32, bd += 4 * (256 >> 4)) {
#pragma unroll
          for (int u = 0; u < 4; ++u) tc::mma_ts(tmem + T_P, a + 8 * u, bd + u * (256 >> 4), id128, (ps | s | u) != 0);
        }
      }
    };
    // (a_hi, a_lo: TMEM, 64 columns) x (b_hi, b_lo: 64-column smem tiles, N rows)^T -> d
    auto issue_t64 = [&](uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo, uint32_t idesc,
                         bool acc) {
#pragma unroll 1
      for (int ps = 0; ps < 3; ++ps) {
        uint32_t a = tmem + (ps == 2 ? a_lo : a_hi);
        uint64_t bd = tc::smem_desc(ps == 1 ? b_lo : b_hi, kLbo, kRg64);
#pragma unroll 1
        for (int s = 0; s < kC / 8; s += 4, a += 32, bd += 4 * ((2 * kLbo) >> 4)) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            tc::mma_ts(tmem + d, a + 8 * u, bd + u * ((2 * kLbo) >> 4), idesc, acc || (ps | s | u) != 0);
        }
      }
    };
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);  // this warp's TMEM lanes
    const bool row_ok = r < dv;
    float *Ap = reinterpret_cast<float *>(sm + OFF_A);
    float *Tp = reinterpret_cast<float *>(sm + OFF_TP);
    float *Yp = reinterpret_cast<float *>(sm + OFF_Y);
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

    for (int c = 0; c < nch; ++c) {
      const ChunkGates &G = gates[c & 1];
      const uint32_t par = c & 1;
      const int nt = min(kC, t1 - t0 - c * kC);
      const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
      // ---- 0: (thread 0) the Gram product once the chunk's operands are stored
      bool ok0 = true;
      if (r == 0 && (ok0 = wait_or_abort(&bars.kq, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue_gram();
        commit(&bars.g, par);
      }
      __syncwarp();
      // ---- 1: split S into the tf32 A operands of P | R, decay S in place
      bool ok = ok0 && (c == 0 || wait_or_abort(&bars.u, par ^ 1, lim, p.status, abort_flag)) &&
                wait_or_abort(&bars.gates, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      const float e_last = G.e_last;
#pragma unroll 1
      for (int q = 0; q < kDK / 16; ++q) {
        uint32_t v[16], hi[16], lo[16];
        tc::tmem_ld16(tl + T_S + 16 * q, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float s = __uint_as_float(v[e]);
          tc::split_tf32(s, hi[e], lo[e]);
          v[e] = __float_as_uint(s * e_last);
        }
        tc::tmem_st16(tl + T_SHI + 16 * q, hi);
        tc::tmem_st16(tl + T_SLO + 16 * q, lo);
        tc::tmem_st16(tl + T_S + 16 * q, v);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars.split);

      // v_t[r] of this chunk, in flight while A and B are formed
      float x[kC];
#pragma unroll
      for (int t = 0; t < kC; ++t)
        x[t] = (t < nt && row_ok) ? __ldg(p.v + ((tb + t) * p.Hv + h) * dv + r) : 0.f;

      // ---- 2: row r of A (r < 64: A_rj = b_r Gam(j,r) G_rj, j < r, packed
      // to smem) or of B (r >= 64: B_tj = Gam(j,t) M_jt, j <= t, t = r - 64,
      // kept in registers until its operand tile is free), from the Gram
      // accumulator's lane r (k_r.k_j for r < 64, q_t.k_j for r >= 64)
      ok = ok0 && wait_or_abort(&bars.g, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      float brow[kC];
      {
        const int t = r < kC ? r : r - kC;
        const float ct = G.cum[t], bt = G.beta[t];
        const int st = G.seg[t], nt_neg = G.nneg[t];
        ld64(tl + T_R, brow);  // the Gram row, weighted in place
        tc::fence_before_sync();
        mbar_arrive(&bars.ab);  // the Gram columns are read: free for R
#pragma unroll
        for (int j = 0; j < kC; ++j) {
          const float m = ex2(ct - G.cum[j]);
          const float gm = st > j ? 0.f : (((nt_neg - G.nneg[j]) & 1) ? -m : m);  // Gam(j, t) for j <= t
          brow[j] *= gm;
        }
        if (r < kC) {
          float *arow = Ap + a_row(t);
#pragma unroll
          for (int j4 = 0; j4 < kC; j4 += 4)
            if (j4 < a1_of(t))
              *reinterpret_cast<float4 *>(arow + j4) =
                  make_float4(j4 < t ? bt * brow[j4] : 0.f, j4 + 1 < t ? bt * brow[j4 + 1] : 0.f,
                              j4 + 2 < t ? bt * brow[j4 + 2] : 0.f, j4 + 3 < t ? bt * brow[j4 + 3] : 0.f);
        } else {
#pragma unroll
          for (int j = 0; j < kC; ++j)
            if (j > t) brow[j] = 0.f;
        }
      }
      named_sync_rows();  // A visible to every row thread
      if (r == 0 && (ok0 = wait_or_abort(&bars.split, par, lim, p.status, abort_flag) &&
                           wait_or_abort(&bars.ab, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue_pr();  // P | R = S [K;Q]^T
        commit(&bars.pr, par);
      }
      __syncwarp();

      // ---- 3: T = (I + A)^-1 (fp32, packed), while P | R runs
      invert_unit_lower(Ap, Tp, Yp, r);

      // ---- 4: once P | R is done (the last reader of S hi / lo and of the
      // [K;Q] tiles): X = b o (v - E o P) -> tf32 hi / lo, R <- E o R, T and
      // B -> tf32 operand tiles
      ok = ok0 && wait_or_abort(&bars.pr, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
      {
        float pv[kC];
        ld64(tl + T_P, pv);
#pragma unroll
        for (int t = 0; t < kC; ++t) x[t] = G.beta[t] * (x[t] - G.E[t] * pv[t]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) tc::split_tf32(x[16 * q + e], hi[e], lo[e]);
          tc::tmem_st16(tl + T_XHI + 16 * q, hi);
          tc::tmem_st16(tl + T_XLO + 16 * q, lo);
        }
      }
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t w[16];
        tc::tmem_ld16(tl + T_R + 16 * q, w);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(G.E[16 * q + e] * __uint_as_float(w[e]));
        tc::tmem_st16(tl + T_R + 16 * q, w);
      }
      // T operand: row r / 2, columns 32 (r % 2) .. + 31, from the packed rows
      {
        const int t = r >> 1, j0 = 32 * (r & 1);
        const float *trow = Tp + t_row(t);
#pragma unroll 1
        for (int j4 = j0; j4 < j0 + 32; j4 += 4) {
          // the packed row's slots above the diagonal are never written: zero them here
          float4 v4 = j4 < b1_of(t) ? *reinterpret_cast<const float4 *>(trow + j4) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (j4 > t) v4.x = 0.f;
          if (j4 + 1 > t) v4.y = 0.f;
          if (j4 + 2 > t) v4.z = 0.f;
          if (j4 + 3 > t) v4.w = 0.f;
          sts_split4(sm, OFF_THI + sq_off(t, j4), OFF_TLO + sq_off(t, j4), v4);
        }
      }
      if (r >= kC) {
        const int t = r - kC;
#pragma unroll
        for (int j4 = 0; j4 < kC; j4 += 4)
          sts_split4(sm, OFF_BHI + sq_off(t, j4), OFF_BLO + sq_off(t, j4),
                     make_float4(brow[j4], brow[j4 + 1], brow[j4 + 2], brow[j4 + 3]));
      }
      tc::tmem_wait_st();
      fence_proxy_async_smem();  // T and B written by the generic proxy, read by the MMA
      tc::fence_before_sync();
      mbar_arrive(&bars.xt);
      if (r == 0 && (ok0 = wait_or_abort(&bars.xt, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue_t64(T_D, T_XHI, T_XLO, thi, tlo, id64, false);  // D = X T^T
        commit(&bars.d, par);
      }
      __syncwarp();

      // ---- 5: D -> tf32 hi / lo (A of O and of the update)
      ok = ok0 && wait_or_abort(&bars.d, par, lim, p.status, abort_flag);
      if (named_any_rows(!ok)) break;
      tc::fence_after_sync();
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t w[16], hi[16], lo[16];
        tc::tmem_ld16(tl + T_D + 16 * q, w);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) tc::split_tf32(__uint_as_float(w[e]), hi[e], lo[e]);
        tc::tmem_st16(tl + T_DHI + 16 * q, hi);
        tc::tmem_st16(tl + T_DLO + 16 * q, lo);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(&bars.dd);
      // O (thread 0) and the update (thread 32) are independent products on
      // the same A operand: two issuing threads keep the tensor core fed
      if (r == 0 && (ok0 = wait_or_abort(&bars.dd, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue_t64(T_R, T_DHI, T_DLO, bhi, blo, id64, true);  // O = E o R + D B^T
        commit(&bars.o, par);
      } else if (r == 32 && (ok0 = wait_or_abort(&bars.dd, par, lim, p.status, abort_flag) &&
                                   wait_or_abort(&bars.kt, par, lim, p.status, abort_flag))) {
        tc::fence_after_sync();
        issue_t64(T_S, T_DHI, T_DLO, kthi, ktlo, id128, true);  // S += D (F o K)
        commit(&bars.u, par);
      }
      __syncwarp();

      // ---- 6: outputs
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
      named_sync_rows();  // every row has read O: the next Gram may overwrite it
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
    const float *qg = p.q, *kg = p.k;
    // the next chunk's k and q: [token block half][channel block half][token in
    // block]; this thread's 4 x 4 blocks are tokens 4a..4a+3, channels
    // 4b..4b+3 with a = al + 8 ah, b = bl + 4 pw + 16 bh
    float4 kr[2][2][4], qr[2][2][4];
    auto load_rows = [&](const float *src, int c, float4 (&dst)[2][2][4]) {
      const int nt = min(kC, t1 - t0 - c * kC);
      const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int bh = 0; bh < 2; ++bh)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int tok = 4 * (al + 8 * ah) + u, b = bl + 4 * pw + 16 * bh;
            dst[ah][bh][u] = tok < nt ? __ldg(reinterpret_cast<const float4 *>(src + ((tb + tok) * p.Hk + g) * kDK + 4 * b))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
          }
    };
    // token-major rows: k at row j, q at row 64 + j
    auto store_rows = [&](const float4 (&src)[2][2][4], int row0) {
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int bh = 0; bh < 2; ++bh)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = row0 + 4 * (al + 8 * ah) + u, b = bl + 4 * pw + 16 * bh;
            const uint32_t o = (uint32_t)(j / 8) * kKqRg + (uint32_t)b * 128 + (uint32_t)(j % 8) * 16;
            sts_split4(sm, OFF_KQHI + o, OFF_KQLO + o, src[ah][bh][u]);
          }
    };
    // channel-major F o K: K[j][c] F_j at (channel c, token j)
    auto store_kt = [&](const ChunkGates &G) {
#pragma unroll
      for (int ah = 0; ah < 2; ++ah) {
        const int a = al + 8 * ah;
        const float f0 = G.F[4 * a], f1 = G.F[4 * a + 1], f2 = G.F[4 * a + 2], f3 = G.F[4 * a + 3];
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
            const uint32_t o = (uint32_t)(ch / 8) * kRg64 + (uint32_t)a * kLbo + (uint32_t)(ch % 8) * 16;
            sts_split4(sm, OFF_KTHI + o, OFF_KTLO + o, make_float4(col[e][0], col[e][1], col[e][2], col[e][3]));
          }
        }
      }
    };
    // gate scan of chunk c by producer warp 0: two tokens per lane
    auto form_gates = [&](int c) {
      ChunkGates &G = gates[c & 1];
      const int nt = min(kC, t1 - t0 - c * kC);
      const int64_t tb = (int64_t)t0 + (int64_t)c * kC;
      float la[2], bb[2];
      int zi[2], ng[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 2 * lane + e;
        const float a = t < nt ? __ldg(p.alpha + (tb + t) * p.Hv + h) : 1.f;
        bb[e] = t < nt ? __ldg(p.beta + (tb + t) * p.Hv + h) : 0.f;
        la[e] = a != 0.f ? log2f(fabsf(a)) : 0.f;
        zi[e] = a == 0.f ? t : -1;
        ng[e] = a < 0.f ? 1 : 0;
      }
      // inclusive scans over the 64 tokens (lane holds tokens 2 lane, 2 lane + 1)
      float cs = la[0] + la[1];
      int zs = max(zi[0], zi[1]), ns = ng[0] + ng[1];
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const float cu = __shfl_up_sync(0xffffffffu, cs, m);
        const int zu = __shfl_up_sync(0xffffffffu, zs, m), nu = __shfl_up_sync(0xffffffffu, ns, m);
        if (lane >= m) {
          cs += cu;
          zs = max(zs, zu);
          ns += nu;
        }
      }
      // exclusive prefix for this lane's first token
      float cx = __shfl_up_sync(0xffffffffu, cs, 1);
      int nx = __shfl_up_sync(0xffffffffu, ns, 1), zx = __shfl_up_sync(0xffffffffu, zs, 1);
      if (lane == 0) {
        cx = 0.f;
        nx = 0;
        zx = -1;
      }
      G.cum[2 * lane] = cx + la[0];
      G.cum[2 * lane + 1] = cs;
      G.seg[2 * lane] = max(zx, zi[0]);
      G.seg[2 * lane + 1] = zs;
      G.nneg[2 * lane] = nx + ng[0];
      G.nneg[2 * lane + 1] = ns;
      G.beta[2 * lane] = bb[0];
      G.beta[2 * lane + 1] = bb[1];
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 2 * lane + e;
        G.E[t] = gam(G, -1, t);
        G.F[t] = gam(G, t, kC - 1);
      }
      if (lane == 0) G.e_last = gam(G, -1, kC - 1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.gates);
    };

    // Chunk c + 1 is prepared during chunk c: its k and q are loaded first;
    // after P | R (c) its gates are formed; after O (c) (the last reader of
    // the tiles that T and B overlay) the [K; Q] tiles are stored; after the
    // update of chunk c the channel-major F o K.  Every producer waits for
    // the gates of chunk c + 1 before it stores the [K; Q] tiles, so the gate
    // barrier is never two phases ahead of a waiting producer.
    if (nch > 0) {
      load_rows(kg, 0, kr);
      load_rows(qg, 0, qr);
      if (pw == 0) form_gates(0);
      if (wait_or_abort(&bars.gates, 0, lim, p.status, abort_flag)) {
        store_rows(kr, 0);
        store_rows(qr, kC);
        fence_proxy_async_smem();
        mbar_arrive(&bars.kq);
        store_kt(gates[0]);
        fence_proxy_async_smem();
        mbar_arrive(&bars.kt);
      }
    }
    for (int c = 0; c + 1 < nch && !*abort_flag; ++c) {
      const uint32_t par = c & 1, npar = par ^ 1;
      load_rows(kg, c + 1, kr);
      load_rows(qg, c + 1, qr);
      if (!wait_or_abort(&bars.pr, par, lim, p.status, abort_flag)) break;
      if (pw == 0) form_gates(c + 1);
      if (!wait_or_abort(&bars.gates, npar, lim, p.status, abort_flag) ||
          !wait_or_abort(&bars.o, par, lim, p.status, abort_flag))
        break;
      store_rows(kr, 0);
      store_rows(qr, kC);
      fence_proxy_async_smem();
      mbar_arrive(&bars.kq);
      if (!wait_or_abort(&bars.u, par, lim, p.status, abort_flag)) break;
      store_kt(gates[npar]);
      fence_proxy_async_smem();
      mbar_arrive(&bars.kt);
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
