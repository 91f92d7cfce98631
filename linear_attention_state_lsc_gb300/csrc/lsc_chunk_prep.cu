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
//               to the record), inverts I + A by 16 x 16 blocks and writes the
//               rows of T' = T diag(b), then E, F and e_last.
// Gam is formed from a per-chunk running sum of log2|a| (zeros and signs of a
// tracked apart), so no product of gates under- or overflows on the way.
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
__host__ __device__ constexpr int a_row(int t) { return 4 * quarter_sum(t + 2); }          // sum of a1_of(i), i < t
__host__ __device__ constexpr int t_row(int t) { return 4 * t + 4 * quarter_sum(t - 1); }  // sum of b1_of(i), i < t
static_assert(a_row(1) == 0 && a_row(2) == 4 && a_row(5) == 16 && t_row(1) == 4 && t_row(5) == 4 * 4 + 8, "packing");
static_assert(b1_of(63) == 4 * row_groups(63), "the T' rows written are the packed rows");
constexpr int kAFloats = a_row(kC);
constexpr int kTFloats = t_row(kC);
constexpr int kYFloats = 3 * 16 * 16;  // block-product scratch of the inverse

// gate quantities of one (chunk, v head)
struct Gates {
  float beta[kC];
  float cum[kC];     // running sum of log2|a_t| over the chunk (0 where a_t = 0)
  float E[kC];       // a_0 ... a_t
  float F[kC];       // Gam(t, C-1)
  int32_t seg[kC];   // last t' <= t with a_t' = 0, or -1
  int32_t nneg[kC];  // number of negative a_t' for t' <= t
  float e_last;
  int32_t pad[3];
};

constexpr uint32_t OFF_KQHI = 0;
constexpr uint32_t OFF_KQLO = kKqBytes;
constexpr uint32_t OFF_GRP = 2 * kKqBytes;
constexpr uint32_t G_A = 0;
constexpr uint32_t G_T = G_A + 4 * kAFloats;
constexpr uint32_t G_Y = G_T + 4 * kTFloats;
constexpr uint32_t G_GATES = G_Y + 4 * kYFloats;
constexpr uint32_t kGrpBytes = G_GATES + sizeof(Gates);
constexpr uint32_t OFF_CU = OFF_GRP + kGroups * kGrpBytes;
constexpr uint32_t kSmemBytes = OFF_CU + 4 * (kStagedSeqs + 4);
static_assert(G_T % 16 == 0 && G_Y % 16 == 0 && G_GATES % 16 == 0 && kGrpBytes % 16 == 0, "alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget (one CTA per SM)");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));  // results below 2^-126 flush to 0
  return y;
}

// Gam(j, t) for j <= t (j = -1: E_t)
__device__ __forceinline__ float gam(const Gates &G, int j, int t) {
  if (G.seg[t] > j) return 0.f;
  const float c0 = j >= 0 ? G.cum[j] : 0.f;
  const int n0 = j >= 0 ? G.nneg[j] : 0;
  const float m = ex2(G.cum[t] - c0);
  return ((G.nneg[t] - n0) & 1) ? -m : m;
}

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
__device__ __forceinline__ void fma4(float4 &acc, float s, const float4 &v) {
  acc.x = fmaf(s, v.x, acc.x);
  acc.y = fmaf(s, v.y, acc.y);
  acc.z = fmaf(s, v.z, acc.z);
  acc.w = fmaf(s, v.w, acc.w);
}

// T = (I + A)^-1 by 16 x 16 blocks, on one solver group's 128 threads (A
// packed by rows at Ap; rows and the diagonal of T packed by rows at Tp; Y is
// scratch):
//   diagonal blocks:  T_bb = (I + A_bb)^-1 by forward substitution, thread
//                     16 b + jj forming column jj of T_bb;
//   level L = 1..3:   Y_ab = sum_(b<=m<a) A_am T_mb, then T_ab = -T_aa Y_ab,
//                     for a = b + L; one work item = (block, row, 4 columns).
// Row offsets inside a 16-row block: the rows 16 m + i of a packed triangle
// start at row(16 m) + 16 m i + row(i) (each row of the block is 16 m longer
// than row i of the first block), so only row(16 m) is formed at run time.
__device__ __forceinline__ void invert_unit_lower(const float *Ap, float *Tp, float *Y, int r, int bar_id) {
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
  group_sync(bar_id);
  float4 *Y4 = reinterpret_cast<float4 *>(Y);
#pragma unroll 1
  for (int L = 1; L < 4; ++L) {
    const int nitems = (4 - L) * 64;
    // Y_ab(i, 4 q .. 4 q + 3) = sum over m in [b, a) and kk of A(16 a + i, 16 m + kk) T(16 m + kk, 16 b + 4 q ..)
#pragma unroll 1
    for (int e = r; e < nitems; e += kGroupThreads) {
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
    group_sync(bar_id);
    // T_ab(i, 4 q ..) = -sum over kk <= i of T(16 a + i, 16 a + kk) Y_ab(kk, 4 q ..)
#pragma unroll 1
    for (int e = r; e < nitems; e += kGroupThreads) {
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
    group_sync(bar_id);
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
__device__ __forceinline__ bool locate(const int32_t *cu, int n_seq, int total, int64_t s, const int32_t *idx,
                                       int num_slots, Located &L) {
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
  const int32_t slot = idx[lo];
  if (slot < 0 || slot >= num_slots) return false;
  L.i = lo;
  L.t0 = t0 + (int)c * kC;
  L.nt = min(kC, t1 - L.t0);
  return true;
}

// Gate scan of one (chunk, v head) by one warp: two tokens per lane.
__device__ __forceinline__ void form_gates(Gates &G, const RecurrentParams &p, int h, const Located &L, int lane) {
  float la[2], bb[2];
  int zi[2], ng[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int t = 2 * lane + e;
    const float a = t < L.nt ? __ldg(p.alpha + (int64_t)(L.t0 + t) * p.Hv + h) : 1.f;
    bb[e] = t < L.nt ? __ldg(p.beta + (int64_t)(L.t0 + t) * p.Hv + h) : 0.f;
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
  const int32_t *cu = p.cu;
  if (p.n_seq <= kStagedSeqs) {
    int32_t *cu_s = reinterpret_cast<int32_t *>(sm + OFF_CU);
    for (int e = tid; e <= p.n_seq; e += kThreads) cu_s[e] = __ldg(p.cu + e);
    cu = cu_s;
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
      if (!locate(cu, p.n_seq, p.total_tokens, s, p.idx, p.num_slots, L)) continue;
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
    float *Yp = reinterpret_cast<float *>(gsm + G_Y);
    Gates &G = *reinterpret_cast<Gates *>(gsm + G_GATES);
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lanes
    const int t = r < kC ? r : r - kC;  // A row (r < 64) or B row
    uint32_t n = 0;
    for (int64_t it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
      const int64_t s = it / p.Hk;
      const int g = (int)(it % p.Hk);
      Located L;
      if (!locate(cu, p.n_seq, p.total_tokens, s, p.idx, p.num_slots, L)) continue;
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
        if (r < 32) form_gates(G, p, h, L, lane);
        group_sync(bar_id);
        {
          // row t of Gam(j, t) o Gram (j <= t), four columns at a time
          const float ct = G.cum[t], bt = G.beta[t];
          const int st = G.seg[t], nt_neg = G.nneg[t];
          float *arow = Ap + a_row(t), *brow = rec + kRecB + t * kC;
#pragma unroll
          for (int j4 = 0; j4 < kC; j4 += 4) {
            float w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = j4 + e;
              const float m = ex2(ct - G.cum[j]);
              const float gm = (st > j || j > t) ? 0.f : (((nt_neg - G.nneg[j]) & 1) ? -m : m);
              w[e] = graw[j] * gm;
            }
            if (r < kC) {  // A_tj = b_t Gam(j,t) k_t.k_j, j < t, packed
              if (j4 < a1_of(t))
                *reinterpret_cast<float4 *>(arow + j4) =
                    make_float4(j4 < t ? bt * w[0] : 0.f, j4 + 1 < t ? bt * w[1] : 0.f, j4 + 2 < t ? bt * w[2] : 0.f,
                                j4 + 3 < t ? bt * w[3] : 0.f);
            } else if (j4 < 4 * row_groups(t)) {  // B_tj = Gam(j,t) q_t.k_j, j <= t, to the record
              *reinterpret_cast<float4 *>(brow + j4) = make_float4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        group_sync(bar_id);
        invert_unit_lower(Ap, Tp, Yp, r, bar_id);
        {
          // T' = T diag(b): row r / 2, columns 32 (r % 2) .. + 31
          const int tt = r >> 1, j0 = 32 * (r & 1);
          const float *trow = Tp + t_row(tt);
          float *dst = rec + kRecT + tt * kC;
#pragma unroll 1
          for (int j4 = j0; j4 < j0 + 32; j4 += 4) {
            if (j4 >= b1_of(tt)) break;
            // the packed row's slots above the diagonal are never written: mask them
            const float4 v4 = mask_above(*reinterpret_cast<const float4 *>(trow + j4), j4, tt);
            *reinterpret_cast<float4 *>(dst + j4) =
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
