// lsc_decode.cuh -- the fused GDN decode kernel of liblsc (strided gather ->
// causal_conv1d_update -> gated delta rule -> in-place scatter), instantiated
// per state dtype in lsc_decode_f32.cu and lsc_decode_bf16.cu.
//
// Sources, cited by page title and section:
//   [VA] "非连续 KV Cache" §5 (state indices -> strided state -> gather -> FLA
//        kernel -> scatter), §6 (causal_conv1d_update, recurrent_gated_delta_rule)
//   [KP] "Kapitsa 源码拆解 05：前缀缓存与模型状态恢复", "Attention 与 Gated
//        DeltaNet 保存的历史不同" (gate, predict S k, correct with v, read with q)
//
// The delta rule S' = a S (I - b k k^T) + b v k^T is applied row by row:
// for row r of S,  u_r = S_r . k,  d_r = b (v_r - a u_r),  S'_r = a S_r + d_r k,
// and o_r = S'_r . q = a (S_r . q) + d_r (k . q).  Each row needs only its own
// elements and the broadcast vectors k, q, so the state streams through shared
// memory once: one HBM read and one HBM write per element.  No tensor cores: a
// decode token is a rank-1 update, about 2 flops per state byte.
#pragma once

#include "lsc_gdn_common.cuh"

namespace lsc {
namespace {

constexpr int kDecodeMaxItems = 512;  // work items per CTA and launch

// Bit-level access to element e of a register array of 16-byte vectors (e is a
// compile-time index after unrolling, so this folds to register moves).
template <typename T> struct VecElem;
template <> struct VecElem<float> {
  __device__ __forceinline__ static uint32_t bits(const uint4 *a, int e) {
    const uint4 &v = a[e >> 2];
    const int w = e & 3;
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
  }
  __device__ __forceinline__ static float get(const uint4 *a, int e) { return __uint_as_float(bits(a, e)); }
  __device__ __forceinline__ static void set_bits(uint4 *a, int e, uint32_t b) {
    uint4 &v = a[e >> 2];
    const int w = e & 3;
    if (w == 0) v.x = b; else if (w == 1) v.y = b; else if (w == 2) v.z = b; else v.w = b;
  }
};
template <> struct VecElem<__nv_bfloat16> {
  __device__ __forceinline__ static uint32_t bits(const uint4 *a, int e) {
    const uint4 &v = a[e >> 3];
    const int w = (e & 7) >> 1;
    const uint32_t word = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
    return (e & 1) ? (word >> 16) : (word & 0xffffu);
  }
  __device__ __forceinline__ static float get(const uint4 *a, int e) { return __uint_as_float(bits(a, e) << 16); }
  __device__ __forceinline__ static void set_bits(uint4 *a, int e, uint32_t b) {
    uint4 &v = a[e >> 3];
    const int w = (e & 7) >> 1;
    uint32_t &word = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
    word = (e & 1) ? ((word & 0x0000ffffu) | (b << 16)) : ((word & 0xffff0000u) | (b & 0xffffu));
  }
};

// Fused decode as a persistent, warp-specialised, pipelined kernel.
//
// Work item = (row i, q/k head g): the G = Hv/Hk v heads that share q/k head g.
// One CTA owns every conv channel of its item (q_g, k_g, and the v channels of
// its G heads), so no two CTAs touch the same conv state.  CTA b processes items
// b, b + grid, ... ; their state tiles (TR rows of one head, <= 32 KiB) stream
// through a ring of NS shared-memory stages.  Three roles:
//  * producer warp (one lane): keeps NS tile loads in flight (cp.async.bulk, a
//    `full` mbarrier per stage); when the tile warps release a stage (`empty`)
//    it bulk-stores the tile back through the page stride and refills the
//    stage once the previous store has left shared memory;
//  * conv warps (kConvThreads): one item ahead of the tile warps, run the conv
//    update of the item's channels -- each thread owns 8-channel groups whose
//    inputs it prefetches two items ahead with cp.async and whose new conv
//    state it writes back with 16-byte stores -- then L2-normalise q and k and
//    leave q, k, v, alpha, beta and k.q in a double-buffered y area
//    (`yfull` / `yempty`);
//  * tile warps (kConsumers): each landed tile in place -- 8 threads per state
//    row on 16-byte vectors: u = S_r.k, w = S_r.q, d = b (v_r - a u),
//    S'_r = a S_r + d k, o_r = a w + d (k.q).
// The conv warps keep clear of the TMA unit, whose queue the 32 KiB tile
// copies fill.  Only the conv and ssm views of a page are addressed.  Every
// mbarrier wait is bounded: on expiry the role records LSC_ERR_DEV_TIMEOUT and
// returns; the other roles' waits then expire in turn, and the producer waits
// (bounded) for every copy it issued before returning.
constexpr int kMaxStages = 8;
constexpr int kConvBufs = 3;  // raw conv-input ring of the conv warps
constexpr int kConsumers = 512;
constexpr int kTileWarps = kConsumers / 32;  // arrivals that release a stage or a y buffer
constexpr int kConvThreads = 96;  // 20 warps in all: 96 registers per thread
constexpr int kDecodeBlock = kConsumers + kConvThreads + 32;
constexpr int kProducer = kConsumers + kConvThreads;
constexpr int64_t kTileBytes = 32 << 10;

template <int DK, typename TS>
struct DecodeShape {
  static constexpr int ES = (int)sizeof(TS);
  static constexpr int EPV = 16 / ES;           // state elements per 16-byte vector
  static constexpr int VPR = DK / EPV;          // vectors per state row
  static constexpr int TPR = VPR < 8 ? VPR : 8; // threads per row
  static constexpr int NV = VPR / TPR;          // vectors per thread per row
  static constexpr int NC = NV * EPV;           // columns per thread
  static constexpr int RPP = kConsumers / TPR;  // rows per pass
  // rows per thread handled together; more than one spills at 96 registers
  static constexpr int RPT = 1;
};

__host__ __device__ inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Tiling and dynamic shared-memory layout, computed identically on both sides.
// y area of an item: q (dk), k (dk), v (G dv), alpha (G), beta (G), k.q (1).
struct DecodeGeom {
  int nch, TR, TPH, TPG, NS, y_ab, y_kq;
  int64_t stage_stride, conv_buf, off_conv, ys_buf, off_ys, off_info, total;
  __host__ __device__ DecodeGeom(int dk, int es, int dv, int G, int W, int esc, int ns) {
    nch = 2 * dk + G * dv;
    const int64_t row_bytes = (int64_t)dk * es;
    TR = (int)(kTileBytes / row_bytes);
    if (TR > dv) TR = dv;
    if (TR < 1) TR = 1;
    TPH = (dv + TR - 1) / TR;
    TPG = G * TPH;
    NS = ns;
    y_ab = nch;
    y_kq = nch + 2 * G;
    stage_stride = align_up((int64_t)TR * row_bytes, 128);
    conv_buf = align_up((int64_t)nch * 2 * W * esc, 128);  // per channel: W-1 state, x, W weights
    off_conv = (int64_t)NS * stage_stride;
    ys_buf = align_up((int64_t)(nch + 2 * G + 1) * 4, 128);
    off_ys = off_conv + kConvBufs * conv_buf;
    off_info = off_ys + 2 * ys_buf;
    total = off_info + 2 * 4 * kDecodeMaxItems;
  }
};

template <int ID, int N>
__device__ __forceinline__ void named_sync() {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(N) : "memory");
}

template <int ID, int N>
__device__ __forceinline__ bool named_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "barrier.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(ID), "n"(N)
      : "memory");
  return r != 0;
}

// TC: conv dtype; CW: conv width when fixed at compile time (0: p.conv_width).
template <int DK, typename TS, typename TC, int CW>
__global__ void __launch_bounds__(kDecodeBlock, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using Sh = DecodeShape<DK, TS>;
  using EC = Elem<TC>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], yfull[2], yempty[2];
  __shared__ float red[3][kConvThreads / 32];

  const int tid = threadIdx.x;
  const int W = CW ? CW : p.conv_width, C = p.conv_dim, dv = p.dv, G = p.group, Hk = p.Hk;
  constexpr int esc = (int)sizeof(TC);
  const bool vec = CW != 0 && p.conv_vec != 0;
  const DecodeGeom D(DK, Sh::ES, dv, G, W, esc, p.stages);
  const int NS = D.NS;
  const int n_items = p.n * Hk;
  const int b = blockIdx.x, grid = gridDim.x;
  const int my_items = b < n_items ? (n_items - b + grid - 1) / grid : 0;
  const int my_tiles = my_items * D.TPG;
  int32_t *info_slot = reinterpret_cast<int32_t *>(smem + D.off_info);
  int32_t *info_warm = info_slot + kDecodeMaxItems;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTileWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&yfull[s], 1);
      mbar_init(&yempty[s], kTileWarps);
    }
    fence_mbar_init();
  }

  // rows of this CTA's items: slot (or -1) and warm, loaded once
  auto load_rows = [&]() {
    for (int k = tid; k < my_items; k += kDecodeBlock) {
      const int i = (b + k * grid) / Hk;
      const int32_t slot = p.idx[i];
      const bool ok = slot >= 0 && slot < p.num_slots;
      if (slot >= p.num_slots) report(p.status, LSC_ERR_OUT_OF_RANGE);
      info_slot[k] = ok ? slot : -1;
      info_warm[k] = ok && (p.has_init == nullptr || p.has_init[i] != 0);
    }
    __syncthreads();
  };

  // producer state, shared by the early start below and the producer loop
  int issued_tiles = 0;
  auto tile_addr = [&](int t, uint32_t &bytes, bool &live, bool &load) -> uint8_t * {
    const int k = t / D.TPG, rem = t % D.TPG, hl = rem / D.TPH, rb = rem % D.TPH;
    const int g = (b + k * grid) % Hk;
    const int rows = min(D.TR, dv - rb * D.TR);
    bytes = (uint32_t)rows * DK * Sh::ES;
    const int32_t slot = info_slot[k];
    live = slot >= 0;
    load = live && info_warm[k] != 0;
    if (!live) return nullptr;
    return p.layer + (int64_t)slot * p.page + p.ssm_off +
           (((int64_t)(g * G + hl) * dv + (int64_t)rb * D.TR) * DK) * Sh::ES;
  };
  // the state is read and written once per launch: evict it from L2 first
  // (3 % faster on the fp32 serving-step decode than the default policy)
  auto issue_tile = [&](int t, uint64_t l2_once) {
    if (t >= my_tiles) return;
    uint32_t bytes;
    bool live, load;
    const uint8_t *src = tile_addr(t, bytes, live, load);
    mbar_arrive_expect_tx(&full[t % NS], load ? bytes : 0u);
    if (load) bulk_g2s(smem + (int64_t)(t % NS) * D.stage_stride, src, bytes, &full[t % NS], l2_once);
    issued_tiles = t + 1;
  };

  // Early start (the caller vouches that the previous kernel of the stream
  // writes neither idx, has_init nor this layer's ssm state): read the rows and
  // fill the ring with the first state tiles while that kernel finishes; when
  // the ring holds less than two items, the next item's tiles are prefetched
  // into L2 as well (serving-step decode, fp32 state: 47.6 -> 46.2 us per
  // launch; with a ring of three bf16 items it cost 1 %).  Every other input is
  // read after griddep_wait() as usual.
  const bool early = p.early_state != 0;
  if (early) {
    load_rows();
    if (tid == kProducer) {
      for (int t = 0; t < NS; ++t) issue_tile(t, l2_evict_first_policy());
      const int l2_end = NS < 2 * D.TPG ? min(my_tiles, NS + D.TPG) : NS;
      for (int t = NS; t < l2_end; ++t) {
        uint32_t bytes;
        bool live, load;
        const uint8_t *src = tile_addr(t, bytes, live, load);
        if (load) bulk_prefetch_l2(src, bytes);
      }
    }
  }
  // the previous kernel of the stream may still be running until here
  griddep_wait();
  if (tid == 0) griddep_launch_dependents();
  if (!early) load_rows();

  if (tid >= kProducer) {
    // ------------------------------------------------------------ producer
    if (tid != kProducer) return;
    const uint64_t l2_once = l2_evict_first_policy();
    auto drain = [&](int t_from) {
      report(p.status, LSC_ERR_DEV_TIMEOUT);
      for (int tt = t_from; tt < issued_tiles; ++tt) mbar_wait_bounded(&full[tt % NS], (tt / NS) & 1, p.drain_limit_ns);
      bulk_wait_read_all();
    };
    if (!early)
      for (int t = 0; t < NS; ++t) issue_tile(t, l2_once);
    for (int t = 0; t < my_tiles; ++t) {
      if (!mbar_wait_bounded(&empty[t % NS], (t / NS) & 1, p.wait_limit_ns)) {
        drain(t);
        return;
      }
      uint32_t bytes;
      bool live, load;
      uint8_t *dst = tile_addr(t, bytes, live, load);
      if (live) bulk_s2g(dst, smem + (int64_t)(t % NS) * D.stage_stride, bytes, l2_once);
      bulk_commit();
      // refill the previous tile's stage once its store has left shared memory
      if (t >= 1 && t - 1 + NS < my_tiles) {
        bulk_wait_read_one();
        issue_tile(t - 1 + NS, l2_once);
      }
    }
    bulk_wait_read_all();
    return;
  }

  if (tid >= kConsumers) {
    // ------------------------------------------------------------ conv warps
    const int ct = tid - kConsumers;
    // Vector path (conv width fixed at compile time, 16-byte aligned channel
    // groups): thread ct owns the 8-channel groups ct, ct + kConvThreads, ...;
    // it prefetches each group's conv state, x and weights two items ahead with
    // cp.async into its own slots of a kConvBufs-deep ring, reads them back
    // itself, and writes the group's new conv state straight to the page.
    // Other shapes read the conv inputs from global memory channel by channel.
    constexpr int WW = CW ? CW : 2;
    constexpr int NSV = 8 * (WW - 1) * esc / 16, NXV = 8 * esc / 16, NWV = 8 * WW * esc / 16;
    constexpr int NGV = NSV + NXV + NWV;  // 16-byte vectors of one group
    static_assert(CW == 0 || (8 * (WW - 1) * esc % 16 == 0 && 8 * WW * esc % 16 == 0), "vector conv layout");
    auto first_channel = [&](int g, int cl0) {
      return cl0 < DK ? g * DK + cl0 : (cl0 < 2 * DK ? Hk * DK + g * DK + (cl0 - DK) : 2 * Hk * DK + g * G * dv + (cl0 - 2 * DK));
    };
    auto prefetch = [&](int k) {
      if (vec && k < my_items && info_slot[k] >= 0) {
        const int j = b + k * grid, i = j / Hk, g = j % Hk;
        const bool warm = info_warm[k] != 0;
        const uint8_t *page = p.layer + (int64_t)info_slot[k] * p.page;
        uint8_t *buf = smem + D.off_conv + (k % kConvBufs) * D.conv_buf;
        for (int grp = ct; grp < D.nch / 8; grp += kConvThreads) {
          const int c = first_channel(g, grp * 8);
          uint8_t *dst = buf + (int64_t)grp * NGV * 16;
          if (warm)
            for (int v = 0; v < NSV; ++v) cp_async16(dst + v * 16, page + (int64_t)c * (WW - 1) * esc + v * 16);
          for (int v = 0; v < NXV; ++v)
            cp_async16(dst + (NSV + v) * 16, (const uint8_t *)p.x + ((int64_t)i * C + c) * esc + v * 16);
          for (int v = 0; v < NWV; ++v)
            cp_async16(dst + (NSV + NXV + v) * 16, (const uint8_t *)p.w + (int64_t)c * WW * esc + v * 16);
        }
      }
      cp_async_commit();  // one group per item, empty or not
    };
    prefetch(0);
    prefetch(1);
    // alpha and beta of the next item, loaded one item ahead (threads < 2G)
    auto load_ab = [&](int k) -> float {
      if (ct >= 2 * G || k >= my_items) return 0.f;
      const int j = b + k * grid, i = j / Hk, g = j % Hk;
      const float *src = ct < G ? p.alpha : p.beta;
      return src[(int64_t)i * p.Hv + g * G + (ct % G)];
    };
    float ab_next = load_ab(0);
    for (int k = 0; k < my_items; ++k) {
      const int j = b + k * grid, i = j / Hk, g = j % Hk;
      const int32_t slot = info_slot[k];
      const bool valid = slot >= 0;
      const bool warm = info_warm[k] != 0;
      uint8_t *page = valid ? p.layer + (int64_t)slot * p.page : nullptr;
      const uint8_t *cb = smem + D.off_conv + (k % kConvBufs) * D.conv_buf;
      float *ys = reinterpret_cast<float *>(smem + D.off_ys + (k & 1) * D.ys_buf);
      const float ab = ab_next;
      ab_next = load_ab(k + 1);
      prefetch(k + 2);
      cp_async_wait<2>();  // this thread's copies of item k have landed
      const bool ok = k < 2 || mbar_wait_bounded(&yempty[k & 1], ((k - 2) >> 1) & 1, p.wait_limit_ns);
      if (named_any<2, kConvThreads>(!ok)) {
        if (ct == 0) report(p.status, LSC_ERR_DEV_TIMEOUT);
        cp_async_wait<0>();
        return;
      }
      float sq = 0.f, sk = 0.f, sqk = 0.f;  // partial sums of this thread's q, k channels
      if (valid) {
        if (vec) {
          using VE = VecElem<TC>;
          for (int grp = ct; grp < D.nch / 8; grp += kConvThreads) {
            const int cl0 = grp * 8;
            const uint4 *gp = reinterpret_cast<const uint4 *>(cb + (int64_t)grp * NGV * 16);
            uint4 sv[NSV], xv[NXV], wv[NWV];
#pragma unroll
            for (int v = 0; v < NSV; ++v) sv[v] = warm ? gp[v] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int v = 0; v < NXV; ++v) xv[v] = gp[NSV + v];
#pragma unroll
            for (int v = 0; v < NWV; ++v) wv[v] = gp[NSV + NXV + v];
            uint4 nv[NSV];
            float y[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              float acc = 0.f;
#pragma unroll
              for (int jj = 0; jj < WW - 1; ++jj) acc = fmaf(VE::get(wv, c * WW + jj), VE::get(sv, c * (WW - 1) + jj), acc);
              acc = fmaf(VE::get(wv, c * WW + WW - 1), VE::get(xv, c), acc);
              y[c] = __fdividef(acc, 1.f + __expf(-acc));  // SiLU
              // new conv state = window shifted by one: old taps 1..W-2, then x
#pragma unroll
              for (int jj = 0; jj < WW - 1; ++jj)
                VE::set_bits(nv, c * (WW - 1) + jj, jj < WW - 2 ? VE::bits(sv, c * (WW - 1) + jj + 1) : VE::bits(xv, c));
            }
            uint4 *gst = reinterpret_cast<uint4 *>(page + (int64_t)first_channel(g, cl0) * (WW - 1) * esc);
#pragma unroll
            for (int v = 0; v < NSV; ++v) gst[v] = nv[v];
            float4 *yp = reinterpret_cast<float4 *>(ys + cl0);
            yp[0] = make_float4(y[0], y[1], y[2], y[3]);
            yp[1] = make_float4(y[4], y[5], y[6], y[7]);
            if (cl0 < 2 * DK) {
              float acc2 = 0.f;
#pragma unroll
              for (int c = 0; c < 8; ++c) acc2 = fmaf(y[c], y[c], acc2);
              if (cl0 < DK) sq += acc2;
              else sk += acc2;
            }
          }
        } else {
          // any conv width or alignment: one channel at a time from global memory
          for (int cl = ct; cl < D.nch; cl += kConvThreads) {
            const int c = first_channel(g, cl);
            float win[kMaxTaps];
#pragma unroll
            for (int jj = 0; jj < kMaxTaps - 1; ++jj) win[jj] = (jj < W - 1 && warm) ? EC::ld(page, (int64_t)c * (W - 1) + jj) : 0.f;
            const float xv = EC::ld(p.x, (int64_t)i * C + c);
            float acc = 0.f;
#pragma unroll
            for (int jj = 0; jj < kMaxTaps; ++jj)
              if (jj < W) acc = fmaf(EC::ld(p.w, (int64_t)c * W + jj), jj == W - 1 ? xv : win[jj], acc);
            const float y = __fdividef(acc, 1.f + __expf(-acc));  // SiLU
            ys[cl] = y;
            if (cl < DK) sq = fmaf(y, y, sq);
            else if (cl < 2 * DK) sk = fmaf(y, y, sk);
#pragma unroll
            for (int jj = 0; jj < kMaxTaps - 1; ++jj)
              if (jj < W - 1) EC::st(page, (int64_t)c * (W - 1) + jj, jj < W - 2 ? win[jj + 1] : xv);
          }
        }
        if (ct < 2 * G) ys[D.y_ab + ct] = ab;
      }
      named_sync<2, kConvThreads>();  // raw y written
      if (valid) {
        // k . q needs the q and k channels of every thread
        for (int c = ct; c < DK; c += kConvThreads) sqk = fmaf(ys[c], ys[DK + c], sqk);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
          sq += __shfl_xor_sync(0xffffffffu, sq, m);
          sk += __shfl_xor_sync(0xffffffffu, sk, m);
          sqk += __shfl_xor_sync(0xffffffffu, sqk, m);
        }
        if ((ct & 31) == 0) {
          red[0][ct >> 5] = sq;
          red[1][ct >> 5] = sk;
          red[2][ct >> 5] = sqk;
        }
        named_sync<2, kConvThreads>();
        sq = sk = sqk = 0.f;
#pragma unroll
        for (int w = 0; w < kConvThreads / 32; ++w) {
          sq += red[0][w];
          sk += red[1][w];
          sqk += red[2][w];
        }
        const float inv_q = 1.f / sqrtf(sq + 1e-6f);
        const float inv_k = 1.f / sqrtf(sk + 1e-6f);
        // the raw q, k were last read before the barrier above: scale in place
        for (int c = ct; c < 2 * DK; c += kConvThreads) ys[c] *= c < DK ? inv_q : inv_k;
        if (ct == 0) ys[D.y_kq] = sqk * inv_q * inv_k;
        named_sync<2, kConvThreads>();
      }
      if (ct == 0) mbar_arrive(&yfull[k & 1]);
    }
    cp_async_wait<0>();
    return;
  }

  // -------------------------------------------------------------- tile warps
  // Each warp runs on its own: it waits for y and for each tile itself and
  // releases them with one arrival per warp, so no CTA-wide barrier paces the
  // tile loop and the warps drift apart, hiding one another's latencies.
  constexpr int NP = Sh::EPV / 2;  // float pairs per 16-byte vector
  const int lr = tid % Sh::TPR, lane = tid & 31;
  int t = 0;
  for (int k = 0; k < my_items; ++k) {
    const int j = b + k * grid, i = j / Hk, g = j % Hk;
    const bool valid = info_slot[k] >= 0;
    const bool warm = info_warm[k] != 0;
    const float *ys = reinterpret_cast<const float *>(smem + D.off_ys + (k & 1) * D.ys_buf);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&yfull[k & 1], (k >> 1) & 1, p.wait_limit_ns))) {
      if (lane == 0) report(p.status, LSC_ERR_DEV_TIMEOUT);
      return;
    }
    float kq = 0.f;
    uint64_t k2[Sh::NC / 2], q2[Sh::NC / 2];  // this thread's columns of k and q, in pairs
    if (valid) {
      kq = ys[D.y_kq];
#pragma unroll
      for (int jj = 0; jj < Sh::NV; ++jj) {
        const int c0v = (jj * Sh::TPR + lr) * Sh::EPV;
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          q2[jj * NP + e] = *reinterpret_cast<const uint64_t *>(ys + c0v + 2 * e);
          k2[jj * NP + e] = *reinterpret_cast<const uint64_t *>(ys + DK + c0v + 2 * e);
        }
      }
    }
    for (int tl = 0; tl < D.TPG; ++tl, ++t) {
      const int stage = t % NS;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[stage], (t / NS) & 1, p.wait_limit_ns))) {
        if (lane == 0) report(p.status, LSC_ERR_DEV_TIMEOUT);
        return;
      }
      const int hl = tl / D.TPH, rb = tl % D.TPH;
      const int rows = min(D.TR, dv - rb * D.TR);
      TS *S = reinterpret_cast<TS *>(smem + (int64_t)stage * D.stage_stride);
      float *o = p.out + ((int64_t)i * p.Hv + g * G + hl) * dv + (int64_t)rb * D.TR;
      if (valid) {
        const float a = ys[D.y_ab + hl], bb = ys[D.y_ab + G + hl];
        const uint64_t a2 = f2_pack(a, a);
        const float *vs = ys + 2 * DK + hl * dv + rb * D.TR;
        const int npass = (rows + Sh::RPP * Sh::RPT - 1) / (Sh::RPP * Sh::RPT);
        for (int ps = 0; ps < npass; ++ps) {
          uint4 sv[Sh::RPT][Sh::NV];  // rows kept packed; unpacked on the fly
          float u[Sh::RPT], wq[Sh::RPT];
          int rr[Sh::RPT];
          bool rv[Sh::RPT];
#pragma unroll
          for (int q = 0; q < Sh::RPT; ++q) {
            const int r0 = (ps * Sh::RPT + q) * Sh::RPP + tid / Sh::TPR;
            rv[q] = r0 < rows;
            rr[q] = rv[q] ? r0 : 0;
#pragma unroll
            for (int jj = 0; jj < Sh::NV; ++jj)
              sv[q][jj] = warm ? *reinterpret_cast<const uint4 *>(S + (int64_t)rr[q] * DK + (jj * Sh::TPR + lr) * Sh::EPV)
                               : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int q = 0; q < Sh::RPT; ++q) {
            uint64_t u2 = 0, w2 = 0;  // (even, odd) column partial sums of S_r.k and S_r.q
#pragma unroll
            for (int jj = 0; jj < Sh::NV; ++jj) {
              uint64_t f[NP];
              StatePairs<TS>::unpack(sv[q][jj], f);
#pragma unroll
              for (int e = 0; e < NP; ++e) {
                u2 = f2_fma(f[e], k2[jj * NP + e], u2);
                w2 = f2_fma(f[e], q2[jj * NP + e], w2);
              }
            }
            float ul, uh, wl, wh;
            f2_unpack(u2, ul, uh);
            f2_unpack(w2, wl, wh);
            u[q] = ul + uh;
            wq[q] = wl + wh;
          }
#pragma unroll
          for (int m = Sh::TPR / 2; m >= 1; m >>= 1) {
#pragma unroll
            for (int q = 0; q < Sh::RPT; ++q) {
              u[q] += __shfl_xor_sync(0xffffffffu, u[q], m);
              wq[q] += __shfl_xor_sync(0xffffffffu, wq[q], m);
            }
          }
#pragma unroll
          for (int q = 0; q < Sh::RPT; ++q) {
            const float d = bb * ((rv[q] ? vs[rr[q]] : 0.f) - a * u[q]);
            if (rv[q]) {
              const uint64_t d2 = f2_pack(d, d);
#pragma unroll
              for (int jj = 0; jj < Sh::NV; ++jj) {
                uint64_t f[NP];
                StatePairs<TS>::unpack(sv[q][jj], f);
#pragma unroll
                for (int e = 0; e < NP; ++e) f[e] = f2_fma(a2, f[e], f2_mul(d2, k2[jj * NP + e]));
                *reinterpret_cast<uint4 *>(S + (int64_t)rr[q] * DK + (jj * Sh::TPR + lr) * Sh::EPV) =
                    StatePairs<TS>::pack(f);
              }
              if (lr == 0) o[rr[q]] = fmaf(a, wq[q], d * kq);
            }
          }
        }
      } else {
        for (int r = tid; r < rows; r += kConsumers) o[r] = 0.f;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (lane == 0) mbar_arrive(&yempty[k & 1]);  // after the last tile's __syncwarp: this warp is done with y
  }
}

template <int DK, typename TS, typename TC, int CW>
int launch_decode_t(const DecodeParams &p0, cudaStream_t stream) {
  DecodeParams p = p0;
  const int esc = (int)sizeof(TC);
  // the opt-in shared-memory limit of a block, per device
  static PerDeviceInt optin_limit;
  const int optin = optin_limit.get([](int dev) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return v;
  });
  if (optin <= 0) return LSC_ERR_CUDA;
  const DecodeGeom probe(DK, (int)sizeof(TS), p.dv, p.group, p.conv_width, esc, 0);
  const int64_t fixed = probe.total + 1024;  // conv, y and item buffers, static shared memory
  int64_t ns = (optin - fixed) / probe.stage_stride;
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return LSC_ERR_UNSUPPORTED;
  p.stages = (int)ns;
  const DecodeGeom D(DK, (int)sizeof(TS), p.dv, p.group, p.conv_width, esc, p.stages);
  static SmemLimit limit;  // per instantiation and device
  if (limit.ensure((const void *)decode_kernel<DK, TS, TC, CW>, (int)D.total) != cudaSuccess) {
    cudaGetLastError();
    return LSC_ERR_UNSUPPORTED;
  }
  // one CTA per SM; rows are split into launches so that no CTA holds more than
  // kDecodeMaxItems items
  const int grid_max = p.num_sms;
  const int rows_per_launch = (int)((int64_t)kDecodeMaxItems * grid_max / p.Hk);
  for (int r0 = 0; r0 < p0.n; r0 += rows_per_launch) {
    DecodeParams q = p;
    q.n = min(rows_per_launch, p0.n - r0);
    q.idx = p0.idx + r0;
    q.has_init = p0.has_init ? p0.has_init + r0 : nullptr;
    q.x = (const uint8_t *)p0.x + (int64_t)r0 * p0.conv_dim * esc;
    q.alpha = p0.alpha + (int64_t)r0 * p0.Hv;
    q.beta = p0.beta + (int64_t)r0 * p0.Hv;
    q.out = p0.out + (int64_t)r0 * p0.Hv * p0.dv;
    const int64_t items = (int64_t)q.n * q.Hk;
    const int grid = (int)(items < grid_max ? items : grid_max);
    // programmatic stream serialisation: this grid's CTAs may be placed on SMs
    // as the previous kernel's CTAs leave them (the kernel waits for that
    // kernel's completion before its first global access)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecodeBlock);
    cfg.dynamicSmemBytes = (size_t)D.total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_kernel<DK, TS, TC, CW>, q) != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
  }
  return LSC_OK;
}

// All decode instantiations for one state dtype TS.
template <typename TS>
int launch_decode_ts(const DecodeParams &p, int dk, cudaStream_t s) {
  const bool cbf = p.conv_bf16 != 0;
  const bool w4 = p.conv_width == 4;
#define LSC_DECODE_DK(DKV)                                                                     \
  case DKV:                                                                                    \
    if (cbf)                                                                                   \
      return w4 ? launch_decode_t<DKV, TS, __nv_bfloat16, 4>(p, s)                             \
                : launch_decode_t<DKV, TS, __nv_bfloat16, 0>(p, s);                            \
    return w4 ? launch_decode_t<DKV, TS, float, 4>(p, s) : launch_decode_t<DKV, TS, float, 0>(p, s);
  switch (dk) {
    LSC_DECODE_DK(16)
    LSC_DECODE_DK(32)
    LSC_DECODE_DK(64)
    LSC_DECODE_DK(128)
    default: return LSC_ERR_UNSUPPORTED;
  }
#undef LSC_DECODE_DK
}

}  // namespace
}  // namespace lsc
