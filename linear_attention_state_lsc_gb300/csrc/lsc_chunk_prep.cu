// lsc_chunk_prep.cu -- the preparation kernel of the chunked gated delta rule:
// for every (64-token chunk, v head) of a resumed prefill it forms, from k, q
// and the gates alone, the quantities that do not depend on the state
// (lsc_chunk.h): T' = (I + A)^-1 diag(b), B, E, F and e_last, and writes them
// to the workspace record of that chunk slot and head.  The state kernel
// (lsc_chunked_tc.cu) then needs only matrix products and elementwise work
// per chunk.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §6 (recurrent_gated_delta_rule, the token recurrence)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with q)
// The pages give the token recurrence only; the chunked form is its algebraic
// rearrangement, exact up to rounding.
//
// One persistent CTA per SM walks the work items (chunk slot, qk head g); the
// v heads g*group .. g*group + group - 1 share the item's k, q and Gram
// products.  384 threads:
//   warps 0-3   operands: load the next item's k and q rows, split them into
//               tf32 hi / lo and store the token-major [K; Q] tile once the
//               previous item's Gram product has read it; thread 0 issues the
//               Gram product [K; Q] K^T (M 128: k rows then q rows, N 64,
//               K 128; three tf32 passes hi.hi + hi.lo + lo.hi) into one of
//               two 64-column TMEM buffers and commits it;
//   warps 4-7,  two solver groups, each taking every other v head of the
//   8-11        item: thread r reads row r of the Gram accumulator (k_r.k_j for
//               r < 64, q_(r-64).k_j above), the group scans the head's gates,
//               forms row r of A (packed in shared memory) or of B (straight
//               to the record), inverts I + A (by 2 x 2 blocks, all four
//               warps) and writes the rows of T' = T diag(b), then E, F and
//               e_last.
// Products of gates are formed in token order (running products along a row,
// product scans for E and F), as the token recurrence applies them: a zero
// gate zeroes what follows, tiny ones fade to zero without a division.
// Every wait is bounded: on expiry the thread records LSC_ERR_DEV_TIMEOUT and
// the CTA stops; the state kernel then reads undefined records, and the call's
// results are unspecified (as its status word says).
#include "lsc_chunk.h"
#include "lsc_gdn_common.cuh"
#include "lsc_tc.h"

namespace lsc {
namespace {

using namespace chunk;

constexpr int kThreads = 384;
constexpr int kProdThreads = 128;
constexpr int kGroups = 2;
constexpr int kGroupThreads = 128;
constexpr uint32_t kTmemCols = 128;  // two Gram buffers of 64 columns
constexpr int kStagedSeqs = 4096;    // cu_seqlens kept in shared memory up to this many sequences

// A and T of one (chunk, v head) in shared memory, fp32, 64 x 64 each: A
// transposed (At[j][t] = A_tj, so the 16 rows of a block column are
// contiguous; row stride kC), T by rows (Tm[t][j]; row stride kTs, which puts
// consecutive rows 4 banks apart, so that 16-byte reads of 8 consecutive rows
// at one column meet no bank twice).
constexpr int kTileFloats = kC * kC;
constexpr int kTs = kC + 4;

// gate quantities of one (chunk, v head)
struct Gates {
  float a[kC];     // a_t (1 past the chunk's tokens)
  float beta[kC];  // b_t (0 past the chunk's tokens)
  float E[kC];     // a_0 ... a_t
  float F[kC];     // Gam(t, C-1) = a_(t+1) ... a_(C-1)
  float e_last;
  int32_t pad[3];
};

constexpr uint32_t OFF_KQHI = 0;
constexpr uint32_t OFF_KQLO = kKqBytes;
constexpr uint32_t OFF_GRP = 2 * kKqBytes;
constexpr uint32_t G_A = 0;
constexpr uint32_t G_T = G_A + 4 * kTileFloats;
constexpr uint32_t G_GATES = G_T + 4 * kC * kTs;
constexpr uint32_t kGrpBytes = G_GATES + sizeof(Gates);
constexpr uint32_t OFF_CU = OFF_GRP + kGroups * kGrpBytes;
constexpr uint32_t OFF_SEQOK = OFF_CU + 4 * (kStagedSeqs + 4);
constexpr uint32_t kSmemBytes = OFF_SEQOK + kStagedSeqs;
static_assert(G_T % 16 == 0 && G_GATES % 16 == 0 && kGrpBytes % 16 == 0, "alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget (one CTA per SM)");

// A solver group (128 threads) synchronises on its own named barrier (1 + its
// index) and leaves with the warp reconverged for the .sync.aligned TMEM
// loads that follow.
__device__ __forceinline__ void group_sync(int id) {
  asm volatile("barrier.sync %0, 128;" ::"r"(id) : "memory");
  __syncwarp();
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, uint64_t limit, int32_t *status,
                                              volatile int *abort_flag) {
  if (mbar_wait_bounded(bar, parity, limit)) return true;
  report(status, LSC_ERR_DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

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

__device__ __forceinline__ float4 mask_above(float4 v, int col0, int row) {  // zero the entries with col > row
  if (col0 > row) v.x = 0.f;
  if (col0 + 1 > row) v.y = 0.f;
  if (col0 + 2 > row) v.z = 0.f;
  if (col0 + 3 > row) v.w = 0.f;
  return v;
}

// T = (I + A)^-1 by the solver group's 128 threads (r = thread index in the
// group), by the 2 x 2 block rule for lower triangular matrices,
//   [P 0; R Q]^-1 = [P^-1 0; -Q^-1 R P^-1  Q^-1],
// applied to 16 x 16 blocks and then to 32 x 32 blocks:
//   (1) the four 16 x 16 diagonal blocks by forward substitution (warp w takes
//       block w, lane l column l mod 16) -- their entries above the diagonal,
//       and the two 16 x 16 blocks above the diagonal inside each 32 x 32
//       half, are written zero, so that the products below run over whole
//       blocks;
//   (2) inside each half: X = A_10 T_00, then T_10 = -T_11 X;
//   (3) the 32 x 32 block: X = A_10 T_00, then T_10 = -T_11 X.
// At holds A transposed (At[j][t] = A_tj, t > j; row stride kC), Tm holds T by
// rows (row stride kTs).  The products X are kept in the 32 x 32 block of Tm
// above the diagonal (rows 0..31, columns 32..63), which is never part of T.
// Step (3) reads the lower half's T_11 by columns: (2) copies it, transposed,
// into the top-left 32 x 32 block of At, whose A entries step (3) no longer
// needs.  Each product is an outer-product loop over its inner index with
// 8-byte shared loads (4 or 8 distinct words per warp: one wavefront each).
__device__ __forceinline__ void invert_unit_lower(float *At, float *Tm, int r, int bar_id) {
  const int w = r >> 5, lane = r & 31;
  {
    const int o = 16 * w, jj = lane & 15;
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = i == jj ? 1.f : 0.f;
#pragma unroll
    for (int ip = 0; ip < 15; ++ip) {
      const float *col = At + (o + ip) * kC + o;  // col[i] = A[o + i][o + ip]
#pragma unroll
      for (int i = ip + 1; i < 16; ++i) y[i] = fmaf(-col[i], y[ip], y[i]);
    }
    if (lane < 16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) Tm[(o + i) * kTs + o + jj] = y[i];
    } else {  // zero blocks: rows 32 q .. + 15, columns 32 q + 16 .. + 15
      const int z = 16 * w + lane - 16, q = z >> 5, row = (z & 31) >> 1;
      float4 *dst = reinterpret_cast<float4 *>(Tm + (32 * q + row) * kTs + 32 * q + 16 + 8 * (z & 1));
      dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  group_sync(bar_id);
  {  // (2) X of half p (rows o + 16 .., columns o ..) to rows 0..15, columns 32 + 16 p ..
    const int p = r >> 6, i = (r & 63) >> 2, j4 = 4 * (r & 3), o = 32 * p;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float a = At[(o + m) * kC + o + 16 + i];
      const float4 t = *reinterpret_cast<const float4 *>(Tm + (o + m) * kTs + o + j4);
      x.x = fmaf(a, t.x, x.x);
      x.y = fmaf(a, t.y, x.y);
      x.z = fmaf(a, t.z, x.z);
      x.w = fmaf(a, t.w, x.w);
    }
    *reinterpret_cast<float4 *>(Tm + i * kTs + 32 + 16 * p + j4) = x;
  }
  group_sync(bar_id);
  {  // (2) T of half p: rows o + 16 + i0 .. + 3, column o + lane mod 16
    const int p = w >> 1, o = 32 * p, j = lane & 15, i0 = 8 * (w & 1) + 4 * (lane >> 4);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m4 = 0; m4 < 16; m4 += 4) {
      float xs[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) xs[u] = Tm[(m4 + u) * kTs + 32 + 16 * p + j];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float4 s = *reinterpret_cast<const float4 *>(Tm + (o + 16 + i0 + e) * kTs + o + 16 + m4);
        acc[e] = fmaf(s.x, xs[0], acc[e]);
        acc[e] = fmaf(s.y, xs[1], acc[e]);
        acc[e] = fmaf(s.z, xs[2], acc[e]);
        acc[e] = fmaf(s.w, xs[3], acc[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      Tm[(o + 16 + i0 + e) * kTs + o + j] = -acc[e];
      // the lower half's T_11 by columns: T[48 + i][32 + j] to At[j][16 + i]
      if (p == 1) At[j * kC + 16 + i0 + e] = -acc[e];
    }
    // ... and its two diagonal blocks: T[32 + 16 b + i][32 + 16 b + m] to At[16 b + m][16 b + i]
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = 4 * r + u, b = e >> 8, i = (e >> 4) & 15, m = e & 15;
      At[(16 * b + m) * kC + 16 * b + i] = Tm[(32 + 16 * b + i) * kTs + 32 + 16 * b + m];
    }
  }
  group_sync(bar_id);
  // (3): thread rows ri, ri + 1 of the 32 x 32 block, columns 2 jg, + 1 and
  // 16 + 2 jg, + 1
  const int ri = 8 * w + 2 * (lane >> 3), jc = 2 * (lane & 7);
  {  // X = A_10 T_00 to rows 0..31, columns 32..63; T_00 is zero in columns
     // 16..31 of rows 0..15
    float x[2][4] = {};
#pragma unroll
    for (int m = 0; m < 32; ++m) {
      const float2 a = *reinterpret_cast<const float2 *>(At + m * kC + 32 + ri);
      const float2 t0 = *reinterpret_cast<const float2 *>(Tm + m * kTs + jc);
      x[0][0] = fmaf(a.x, t0.x, x[0][0]);
      x[0][1] = fmaf(a.x, t0.y, x[0][1]);
      x[1][0] = fmaf(a.y, t0.x, x[1][0]);
      x[1][1] = fmaf(a.y, t0.y, x[1][1]);
      if (m >= 16) {
        const float2 t1 = *reinterpret_cast<const float2 *>(Tm + m * kTs + 16 + jc);
        x[0][2] = fmaf(a.x, t1.x, x[0][2]);
        x[0][3] = fmaf(a.x, t1.y, x[0][3]);
        x[1][2] = fmaf(a.y, t1.x, x[1][2]);
        x[1][3] = fmaf(a.y, t1.y, x[1][3]);
      }
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      *reinterpret_cast<float2 *>(Tm + (ri + e) * kTs + 32 + jc) = make_float2(x[e][0], x[e][1]);
      *reinterpret_cast<float2 *>(Tm + (ri + e) * kTs + 48 + jc) = make_float2(x[e][2], x[e][3]);
    }
  }
  group_sync(bar_id);
  {  // T_10 = -T_11 X to rows 32.., columns 0..31; T_11 (read by columns from
     // At) is zero right of its diagonal, so rows 0..15 of the block stop at
     // inner index 15
    float x[2][4] = {};
    const int mend = w < 2 ? 16 : 32;
#pragma unroll 4
    for (int m = 0; m < mend; ++m) {
      const float2 a = *reinterpret_cast<const float2 *>(At + m * kC + ri);
      const float2 t0 = *reinterpret_cast<const float2 *>(Tm + m * kTs + 32 + jc);
      const float2 t1 = *reinterpret_cast<const float2 *>(Tm + m * kTs + 48 + jc);
      x[0][0] = fmaf(a.x, t0.x, x[0][0]);
      x[0][1] = fmaf(a.x, t0.y, x[0][1]);
      x[0][2] = fmaf(a.x, t1.x, x[0][2]);
      x[0][3] = fmaf(a.x, t1.y, x[0][3]);
      x[1][0] = fmaf(a.y, t0.x, x[1][0]);
      x[1][1] = fmaf(a.y, t0.y, x[1][1]);
      x[1][2] = fmaf(a.y, t1.x, x[1][2]);
      x[1][3] = fmaf(a.y, t1.y, x[1][3]);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      *reinterpret_cast<float2 *>(Tm + (32 + ri + e) * kTs + jc) = make_float2(-x[e][0], -x[e][1]);
      *reinterpret_cast<float2 *>(Tm + (32 + ri + e) * kTs + 16 + jc) = make_float2(-x[e][2], -x[e][3]);
    }
  }
}

// The sequence and chunk of chunk slot s: the largest i with
// slot_base(cu[i], i) <= s (a binary search, valid while cu is
// non-decreasing), then chunk c = s - slot_base(cu[i], i).  False when the
// slot belongs to no chunk, the sequence's cu entries are inconsistent (the
// state kernel skips and reports it) or the sequence is a padding one.
struct Located {
  int i, t0, nt;
};
__device__ __forceinline__ bool locate(const int32_t *cu, const uint8_t *seq_ok, int n_seq, int total, int64_t s,
                                       const int32_t *idx, int num_slots, Located &L) {
  if (n_seq <= 0 || slot_base(cu[0], 0) > s) return false;
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(cu[mid], mid) <= s) lo = mid;
    else hi = mid - 1;
  }
  const int t0 = cu[lo], t1 = cu[lo + 1];
  if (t0 < 0 || t1 < t0 || t1 > total) return false;
  const int64_t c = s - slot_base(t0, lo);
  if (c * kC >= (int64_t)(t1 - t0)) return false;
  if (seq_ok) {
    if (!seq_ok[lo]) return false;
  } else {
    const int32_t slot = idx[lo];
    if (slot < 0 || slot >= num_slots) return false;
  }
  L.i = lo;
  L.t0 = t0 + (int)c * kC;
  L.nt = min(kC, t1 - L.t0);
  return true;
}

// The gates of one (chunk, v head), two tokens per lane (alpha 1 and beta 0
// past the chunk's tokens).
struct GateIn {
  float a[2], b[2];
};
__device__ __forceinline__ GateIn load_gates(const RecurrentParams &p, int h, const Located &L, int lane) {
  GateIn in;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int t = 2 * lane + e;
    in.a[e] = t < L.nt ? __ldg(p.alpha + (int64_t)(L.t0 + t) * p.Hv + h) : 1.f;
    in.b[e] = t < L.nt ? __ldg(p.beta + (int64_t)(L.t0 + t) * p.Hv + h) : 0.f;
  }
  return in;
}

// Gate products of one (chunk, v head) by one warp, two tokens per lane:
// E_t = a_0 ... a_t (an inclusive product scan) and F_t = a_(t+1) ... a_(C-1)
// (= E_(C-1) / E_t, formed as a product so that no zero or underflowed E
// divides).  Products run in token order; a zero gate zeroes what follows it,
// a negative one flips signs, and tiny ones fade to zero, as in the token
// recurrence.
__device__ __forceinline__ void form_gates(Gates &G, const GateIn &in, int lane) {
  // inclusive product over this lane's pair, then over the lanes below
  const float p0 = in.a[0], p01 = in.a[0] * in.a[1];
  float inc = p01;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float up = __shfl_up_sync(0xffffffffu, inc, m);
    if (lane >= m) inc = up * inc;
  }
  float exc = __shfl_up_sync(0xffffffffu, inc, 1);  // product of the lanes below
  if (lane == 0) exc = 1.f;
  // suffix products: the lanes above, then within the pair
  float suf = p01;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float dn = __shfl_down_sync(0xffffffffu, suf, m);
    if (lane + m < 32) suf = suf * dn;
  }
  float above = __shfl_down_sync(0xffffffffu, suf, 1);  // product of the lanes above
  if (lane == 31) above = 1.f;
  G.a[2 * lane] = in.a[0];
  G.a[2 * lane + 1] = in.a[1];
  G.beta[2 * lane] = in.b[0];
  G.beta[2 * lane + 1] = in.b[1];
  G.E[2 * lane] = exc * p0;
  G.E[2 * lane + 1] = exc * p01;
  G.F[2 * lane] = in.a[1] * above;
  G.F[2 * lane + 1] = above;
  if (lane == 31) G.e_last = exc * p01;
  __syncwarp();
}

struct PrepBars {
  uint64_t kq;         // the item's [K; Q] tile is stored (every operand thread)
  uint64_t gfull[2];   // Gram buffer b holds the item's products (MMA commit)
  uint64_t gempty[2];  // Gram buffer b has been read (every solver thread)
};

__global__ void __launch_bounds__(kThreads, 1) chunk_prep_kernel(const __grid_constant__ RecurrentParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ PrepBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // cu_seqlens and whether each sequence's slot is in range, staged once
  const int32_t *cu = p.cu;
  const uint8_t *seq_ok = nullptr;
  if (p.n_seq <= kStagedSeqs) {
    int32_t *cu_s = reinterpret_cast<int32_t *>(sm + OFF_CU);
    uint8_t *ok_s = sm + OFF_SEQOK;
    for (int e = tid; e <= p.n_seq; e += kThreads) cu_s[e] = __ldg(p.cu + e);
    for (int e = tid; e < p.n_seq; e += kThreads) {
      const int32_t slot = __ldg(p.idx + e);
      ok_s[e] = slot >= 0 && slot < p.num_slots;
    }
    cu = cu_s;
    seq_ok = ok_s;
  }
  if (tid == 0) {
    mbar_init(&bars.kq, kProdThreads);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.gfull[b], 1);
      mbar_init(&bars.gempty[b], kGroups * kGroupThreads);
    }
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
  const int64_t n_items = n_slots(p.total_tokens, p.n_seq) * p.Hk;

  if (warp < kProdThreads / 32) {
    // ============================================== operands and the Gram MMA
    const int pw = warp, al = lane & 7, bl = lane >> 3;
    const uint32_t kqhi = smem_u32(sm + OFF_KQHI), kqlo = smem_u32(sm + OFF_KQLO);
    constexpr uint32_t id64 = tc::idesc_tf32(128, 64, false);
    uint64_t *last = nullptr;  // thread 0: the last commit's barrier and phase
    uint32_t last_par = 0, n = 0;
    for (int64_t it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      const int64_t s = it / p.Hk;
      const int g = (int)(it % p.Hk);
      Located L;
      if (!locate(cu, seq_ok, p.n_seq, p.total_tokens, s, p.idx, p.num_slots, L)) continue;
      // this thread's 4 x 4 blocks: tokens 4a..4a+3, channels 4b..4b+3 with
      // a = al + 8 ah, b = bl + 4 pw + 16 bh
      float4 kr[2][2][4], qr[2][2][4];
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int bh = 0; bh < 2; ++bh)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int tok = 4 * (al + 8 * ah) + u, b = bl + 4 * pw + 16 * bh;
            const int64_t off = ((int64_t)(L.t0 + tok) * p.Hk + g) * kDK + 4 * b;
            const bool in = tok < L.nt;
            kr[ah][bh][u] = in ? __ldg(reinterpret_cast<const float4 *>(p.k + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
            qr[ah][bh][u] = in ? __ldg(reinterpret_cast<const float4 *>(p.q + off)) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
      // the tile is free once the previous item's Gram product has read it
      if (n >= 1 && !wait_or_abort(&bars.gfull[(n - 1) & 1], ((n - 1) >> 1) & 1, lim, p.status, abort_flag)) break;
#pragma unroll
      for (int ah = 0; ah < 2; ++ah)
#pragma unroll
        for (int bh = 0; bh < 2; ++bh)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * (al + 8 * ah) + u, c4 = 4 * (bl + 4 * pw + 16 * bh);
            sts_split4(sm, OFF_KQHI + kq_off(j, c4), OFF_KQLO + kq_off(j, c4), kr[ah][bh][u]);
            sts_split4(sm, OFF_KQHI + kq_off(kC + j, c4), OFF_KQLO + kq_off(kC + j, c4), qr[ah][bh][u]);
          }
      fence_proxy_async_smem();
      mbar_arrive(&bars.kq);
      if (tid == 0) {
        const uint32_t b = n & 1;
        if (wait_or_abort(&bars.kq, n & 1, lim, p.status, abort_flag) &&
            (n < 2 || wait_or_abort(&bars.gempty[b], ((n - 2) >> 1) & 1, lim, p.status, abort_flag))) {
          tc::fence_after_sync();
          const uint32_t d = tmem + 64 * b;
          // [K; Q] (128 rows) x K (the first 64 rows)^T; a k step of 8 tf32
          // channels is 256 bytes along the tile (16 in the descriptor)
#pragma unroll
          for (int ps = 0; ps < 3; ++ps) {
            const uint64_t ad = tc::smem_desc(ps == 2 ? kqlo : kqhi, 128, kKqRg);
            const uint64_t bd = tc::smem_desc(ps == 1 ? kqlo : kqhi, 128, kKqRg);
#pragma unroll
            for (int k8 = 0; k8 < kDK / 8; ++k8)
              tc::mma_ss(d, ad + 16 * k8, bd + 16 * k8, id64, (ps | k8) != 0);
          }
          tc::mma_commit(&bars.gfull[b]);
          last = &bars.gfull[b];
          last_par = (n >> 1) & 1;
        }
      }
      __syncwarp();
      ++n;
    }
    // the TMEM is freed below: every product issued must be complete
    if (tid == 0 && last) mbar_wait_bounded(last, last_par, p.drain_limit_ns);
  } else {
    // ============================================== solver groups
    const int grp = (warp - kProdThreads / 32) / 4;
    const int r = tid - kProdThreads - grp * kGroupThreads;  // = Gram row = TMEM lane
    const int bar_id = 1 + grp;
    uint8_t *gsm = sm + OFF_GRP + grp * kGrpBytes;
    float *Ap = reinterpret_cast<float *>(gsm + G_A);
    float *Tp = reinterpret_cast<float *>(gsm + G_T);
    Gates &G = *reinterpret_cast<Gates *>(gsm + G_GATES);
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lanes
    const int t = r < kC ? r : r - kC;  // A row (r < 64) or B row
    uint32_t n = 0;
    for (int64_t it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      const int64_t s = it / p.Hk;
      const int g = (int)(it % p.Hk);
      Located L;
      if (!locate(cu, seq_ok, p.n_seq, p.total_tokens, s, p.idx, p.num_slots, L)) continue;
      // the first head's gates in flight while the Gram product is awaited
      GateIn gin;
      if (r < 32 && grp < p.group) gin = load_gates(p, g * p.group + grp, L, lane);
      if (!wait_or_abort(&bars.gfull[n & 1], (n >> 1) & 1, lim, p.status, abort_flag)) break;
      tc::fence_after_sync();
      float graw[kC];
      ld64(tl + 64 * (n & 1), graw);
      tc::fence_before_sync();
      mbar_arrive(&bars.gempty[n & 1]);
#pragma unroll 1
      for (int u = grp; u < p.group; u += kGroups) {
        const int h = g * p.group + u;
        float *rec = p.ws + (s * p.Hv + h) * (int64_t)kRecFloats;
        if (r < 32) {
          if (u != grp) gin = load_gates(p, h, L, lane);
          form_gates(G, gin, lane);
        }
        group_sync(bar_id);
        {
          // row t of Gam(j, t) o Gram (j <= t): Gam(j, t) = a_(j+1) ... a_t as
          // a running product from j = t down to 0
          const float bt = G.beta[t];
          float *brec = rec + kRecB;
          float w[kC];
          float gm = 1.f;
#pragma unroll
          for (int j = kC - 1; j >= 0; --j) {
            if (j < t) gm *= G.a[j + 1];
            w[j] = j <= t ? graw[j] * gm : 0.f;
          }
          if (r < kC) {  // A_tj = b_t Gam(j,t) k_t.k_j, j < t, transposed
#pragma unroll
            for (int j = 0; j < kC - 1; ++j)
              if (j < t) Ap[j * kC + t] = bt * w[j];
          } else {  // B_tj = Gam(j,t) q_t.k_j, j <= t, to the record
#pragma unroll
            for (int j4 = 0; j4 < kC; j4 += 4)
              if (j4 < 4 * row_groups(t))
                *reinterpret_cast<float4 *>(brec + rec_off(t, j4)) = make_float4(w[j4], w[j4 + 1], w[j4 + 2], w[j4 + 3]);
          }
        }
        group_sync(bar_id);
        invert_unit_lower(Ap, Tp, r, bar_id);
        group_sync(bar_id);
        {
          // T' = T diag(b): row r / 2, columns 32 (r % 2) .. + 31
          const int tt = r >> 1, j0 = 32 * (r & 1);
          const float *trow = Tp + tt * kTs;
          float *dst = rec + kRecT;
#pragma unroll 1
          for (int j4 = j0; j4 < j0 + 32; j4 += 4) {
            if (j4 >= 4 * row_groups(tt)) break;
            // the packed row's slots above the diagonal are never written: mask them
            const float4 v4 = mask_above(*reinterpret_cast<const float4 *>(trow + j4), j4, tt);
            *reinterpret_cast<float4 *>(dst + rec_off(tt, j4)) =
                make_float4(v4.x * G.beta[j4], v4.y * G.beta[j4 + 1], v4.z * G.beta[j4 + 2], v4.w * G.beta[j4 + 3]);
          }
        }
        if (r < kC) {
          rec[kRecE + r] = G.E[r];
          rec[kRecF + r] = G.F[r];
        }
        if (r == 0) rec[kRecMisc] = G.e_last;
        group_sync(bar_id);  // the group's shared memory is reused by its next head
      }
      ++n;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

// Workspace records of every (chunk slot, v head) of the call; p.ws must hold
// workspace_bytes(total_tokens, n_seq, Hv) bytes, 16-byte aligned.
int launch_chunk_prep(const RecurrentParams &p, int num_sms, cudaStream_t s) {
  static SmemLimit limit;
  if (limit.ensure((const void *)chunk_prep_kernel, (int)kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  const int64_t items = n_slots(p.total_tokens, p.n_seq) * p.Hk;
  const int grid = (int)(items < num_sms ? items : num_sms);
  if (grid <= 0) return LSC_OK;
  chunk_prep_kernel<<<grid, kThreads, kSmemBytes, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace lsc
