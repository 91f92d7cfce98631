// lsc_gdn.cu -- GDN kernels of liblsc: the fused decode step (strided gather ->
// causal_conv1d_update -> gated delta rule -> in-place scatter) and the
// token-by-token recurrence of a resumed prefill.
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
// elements and the broadcast vectors k, q, so the state streams through
// registers once: one HBM read and one HBM write per element.  No tensor cores:
// a decode token is a rank-1 update, about 2 flops per state byte.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lsc_internal.h"
#include "lsc_ptx.h"

namespace lsc {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeMaxItems = 512;  // work items per CTA and launch
constexpr int kMaxDv = 128;
constexpr int kMaxTaps = 8;

__device__ __forceinline__ void report(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// Conv-side element access (conv dtype is f32 or bf16, chosen at run time).
__device__ __forceinline__ float ld_conv(const void *base, int64_t i, bool bf16) {
  return bf16 ? bf16_bits_to_float(((const uint16_t *)base)[i]) : ((const float *)base)[i];
}
__device__ __forceinline__ void st_conv(void *base, int64_t i, float v, bool bf16) {
  if (bf16) ((uint16_t *)base)[i] = float_to_bf16_bits(v);
  else ((float *)base)[i] = v;
}

// 16-byte vectors of state elements <-> floats.
template <typename TS> struct StateVec;
template <> struct StateVec<float> {
  __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 pack(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};
template <> struct StateVec<__nv_bfloat16> {
  __device__ __forceinline__ static void unpack(const uint4 &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 pack(const float *f) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);  // .x = low half
      w[k] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Fused decode as a persistent, warp-specialised, TMA-pipelined kernel.
//
// Work item = (row i, q/k head g): the G = Hv/Hk v heads that share q/k head g.
// One CTA owns every conv channel of its item (q_g, k_g, and the v channels of
// its G heads), so no two CTAs touch the same conv state.  CTA b processes items
// b, b + grid, ... ; their state tiles (TR rows of one head, <= 32 KiB) stream
// through a ring of NS shared-memory stages.
//  * Producer warp (one lane): keeps NS tile loads in flight (cp.async.bulk, a
//    `full` mbarrier per stage) and the conv inputs of the next two items in a
//    double buffer; when the consumers release a stage (`empty` mbarrier) it
//    bulk-stores the tile back through the page stride, waits for the store to
//    leave shared memory, and refills the stage.
//  * Consumer warps (kConsumers threads): conv update of the item, L2 norms,
//    then each landed tile in place -- 8 threads per state row on 16-byte
//    vectors: u = S_r.k, w = S_r.q, d = b (v_r - a u), S'_r = a S_r + d k,
//    o_r = a w + d (k.q).
// Only the conv and ssm views of a page are addressed.  Every mbarrier wait is
// bounded: on expiry the CTA records LSC_ERR_DEV_TIMEOUT, the producer waits
// (bounded) for every copy it issued, and the CTA returns.
constexpr int kMaxStages = 8;
constexpr int kConsumers = 512;
constexpr int kDecodeBlock = kConsumers + 32;
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
};

__host__ __device__ inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Tiling and dynamic shared-memory layout, computed identically on both sides.
struct DecodeGeom {
  int nch, TR, TPH, TPG, NS;
  int64_t stage_stride, conv_buf, off_st, off_xs, off_ws, off_conv, ys_buf, off_ys, off_info, total;
  __host__ __device__ DecodeGeom(int dk, int es, int dv, int G, int W, int esc, int ns) {
    nch = 2 * dk + G * dv;
    const int64_t row_bytes = (int64_t)dk * es;
    TR = (int)(kTileBytes / row_bytes);
    if (TR > dv) TR = dv;
    if (TR < 1) TR = 1;
    TPH = (dv + TR - 1) / TR;
    TPG = G * TPH;
    NS = ns;
    stage_stride = align_up((int64_t)TR * row_bytes, 128);
    off_st = 0;
    off_xs = align_up((int64_t)nch * (W - 1) * esc, 16);
    off_ws = off_xs + align_up((int64_t)nch * esc, 16);
    conv_buf = align_up(off_ws + (int64_t)nch * W * esc, 128);
    off_conv = (int64_t)NS * stage_stride;
    ys_buf = align_up((int64_t)(nch + 2 * G) * 4, 128);
    off_ys = off_conv + 2 * conv_buf;
    off_info = off_ys + 2 * ys_buf;
    total = off_info + 2 * 4 * kDecodeMaxItems;
  }
};

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "barrier.red.or.pred p, 1, %2, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsumers)
      : "memory");
  return r != 0;
}

template <int DK, typename TS>
__global__ void __launch_bounds__(kDecodeBlock, 1) decode_kernel(const __grid_constant__ DecodeParams p) {
  using Sh = DecodeShape<DK, TS>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], cfull[2];
  __shared__ float red[3][kConsumers / 32];

  const int tid = threadIdx.x;
  const int W = p.conv_width, C = p.conv_dim, dv = p.dv, G = p.group, Hk = p.Hk;
  const int esc = p.conv_bf16 ? 2 : 4;
  const bool cbf = p.conv_bf16 != 0;
  const bool tma_conv = p.conv_tma != 0;
  const DecodeGeom D(DK, Sh::ES, dv, G, W, esc, p.stages);
  const int NS = D.NS;
  const int n_items = p.n * Hk;
  const int b = blockIdx.x, grid = gridDim.x;
  const int my_items = b < n_items ? (n_items - b + grid - 1) / grid : 0;
  const int my_tiles = my_items * D.TPG;
  int32_t *info_slot = reinterpret_cast<int32_t *>(smem + D.off_info);
  int32_t *info_warm = info_slot + kDecodeMaxItems;

  // rows of this CTA's items: slot (or -1) and warm, loaded once
  for (int k = tid; k < my_items; k += kDecodeBlock) {
    const int i = (b + k * grid) / Hk;
    const int32_t slot = p.idx[i];
    const bool ok = slot >= 0 && slot < p.num_slots;
    if (slot >= p.num_slots) report(p.status, LSC_ERR_OUT_OF_RANGE);
    info_slot[k] = ok ? slot : -1;
    info_warm[k] = ok && (p.has_init == nullptr || p.has_init[i] != 0);
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&cfull[0], 1);
    mbar_init(&cfull[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (tid >= kConsumers) {
    // ------------------------------------------------------------ producer
    if (tid != kConsumers) return;
    int issued_tiles = 0, issued_convs = 0;
    auto issue_conv = [&](int k) {
      if (k >= my_items) return;
      const int j = b + k * grid, i = j / Hk, g = j % Hk;
      const int32_t slot = info_slot[k];
      const bool warm = info_warm[k] != 0;
      uint8_t *buf = smem + D.off_conv + (k & 1) * D.conv_buf;
      const uint32_t bytes = (slot >= 0 && tma_conv) ? (uint32_t)(D.nch * ((warm ? W - 1 : 0) + 1 + W) * esc) : 0u;
      mbar_arrive_expect_tx(&cfull[k & 1], bytes);
      if (bytes) {
        const uint8_t *page = p.layer + (int64_t)slot * p.page;
        const int c0[3] = {g * DK, Hk * DK + g * DK, 2 * Hk * DK + g * G * dv};
        const int cn[3] = {DK, DK, G * dv};
        const int cl0[3] = {0, DK, 2 * DK};
        for (int sgm = 0; sgm < 3; ++sgm) {
          if (warm)
            bulk_g2s(buf + D.off_st + (int64_t)cl0[sgm] * (W - 1) * esc, page + (int64_t)c0[sgm] * (W - 1) * esc,
                     (uint32_t)(cn[sgm] * (W - 1) * esc), &cfull[k & 1]);
          bulk_g2s(buf + D.off_xs + (int64_t)cl0[sgm] * esc, (const uint8_t *)p.x + ((int64_t)i * C + c0[sgm]) * esc,
                   (uint32_t)(cn[sgm] * esc), &cfull[k & 1]);
          bulk_g2s(buf + D.off_ws + (int64_t)cl0[sgm] * W * esc, (const uint8_t *)p.w + (int64_t)c0[sgm] * W * esc,
                   (uint32_t)(cn[sgm] * W * esc), &cfull[k & 1]);
        }
      }
      issued_convs = k + 1;
    };
    // global address of tile t's rows in the state view
    auto tile_addr = [&](int t, uint32_t &bytes, bool &live, bool &load) -> uint8_t * {
      const int k = t / D.TPG, rem = t % D.TPG, hl = rem / D.TPH, rb = rem % D.TPH;
      const int j = b + k * grid, g = j % Hk;
      const int rows = min(D.TR, dv - rb * D.TR);
      bytes = (uint32_t)rows * DK * Sh::ES;
      const int32_t slot = info_slot[k];
      live = slot >= 0;
      load = live && info_warm[k] != 0;
      if (!live) return nullptr;
      return p.layer + (int64_t)slot * p.page + p.ssm_off +
             (((int64_t)(g * G + hl) * dv + (int64_t)rb * D.TR) * DK) * Sh::ES;
    };
    auto issue_tile = [&](int t) {
      if (t >= my_tiles) return;
      uint32_t bytes;
      bool live, load;
      const uint8_t *src = tile_addr(t, bytes, live, load);
      mbar_arrive_expect_tx(&full[t % NS], load ? bytes : 0u);
      if (load) bulk_g2s(smem + (int64_t)(t % NS) * D.stage_stride, src, bytes, &full[t % NS]);
      issued_tiles = t + 1;
    };
    issue_conv(0);
    issue_conv(1);
    for (int t = 0; t < NS; ++t) issue_tile(t);
    for (int t = 0; t < my_tiles; ++t) {
      if (!mbar_wait_bounded(&empty[t % NS], (t / NS) & 1, p.wait_limit_ns)) {
        report(p.status, LSC_ERR_DEV_TIMEOUT);
        for (int tt = t; tt < issued_tiles; ++tt)
          mbar_wait_bounded(&full[tt % NS], (tt / NS) & 1, p.drain_limit_ns);
        for (int kk = issued_convs - 2 < 0 ? 0 : issued_convs - 2; kk < issued_convs; ++kk)
          mbar_wait_bounded(&cfull[kk & 1], (kk >> 1) & 1, p.drain_limit_ns);
        bulk_wait_read_all();
        return;
      }
      uint32_t bytes;
      bool live, load;
      uint8_t *dst = tile_addr(t, bytes, live, load);
      if (live) bulk_s2g(dst, smem + (int64_t)(t % NS) * D.stage_stride, bytes);
      bulk_commit();
      // the consumers have finished an item's conv staging before its first tile
      if (t % D.TPG == 0) issue_conv(t / D.TPG + 2);
      if (t + NS < my_tiles) {
        bulk_wait_read_all();  // tile t's store has left the stage
        issue_tile(t + NS);
      }
    }
    bulk_wait_read_all();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int lr = tid % Sh::TPR;
  int t = 0;
  for (int k = 0; k < my_items; ++k) {
    const int j = b + k * grid, i = j / Hk, g = j % Hk;
    const int32_t slot = info_slot[k];
    const bool valid = slot >= 0;
    const bool warm = info_warm[k] != 0;
    uint8_t *page = valid ? p.layer + (int64_t)slot * p.page : nullptr;
    const uint8_t *cb = smem + D.off_conv + (k & 1) * D.conv_buf;
    float *ys = reinterpret_cast<float *>(smem + D.off_ys + (k & 1) * D.ys_buf);

    // conv update of the item's channels
    if (consumer_any(!mbar_wait_bounded(&cfull[k & 1], (k >> 1) & 1, p.wait_limit_ns))) {
      if (tid == 0) report(p.status, LSC_ERR_DEV_TIMEOUT);
      return;  // the producer drains the copies in flight
    }
    float kq = 0.f;
    float kreg[Sh::NC], qreg[Sh::NC];
    if (valid) {
      for (int cl = tid; cl < D.nch; cl += kConsumers) {
        const int c = cl < DK ? g * DK + cl
                              : (cl < 2 * DK ? Hk * DK + g * DK + (cl - DK) : 2 * Hk * DK + g * G * dv + (cl - 2 * DK));
        float win[kMaxTaps];
        for (int jj = 0; jj < W - 1; ++jj) {
          float v = 0.f;
          if (warm)
            v = tma_conv ? ld_conv(cb + D.off_st, (int64_t)cl * (W - 1) + jj, cbf)
                         : ld_conv(page, (int64_t)c * (W - 1) + jj, cbf);
          win[jj] = v;
        }
        win[W - 1] = tma_conv ? ld_conv(cb + D.off_xs, cl, cbf) : ld_conv(p.x, (int64_t)i * C + c, cbf);
        float z = 0.f;
        for (int jj = 0; jj < W; ++jj)
          z = fmaf(tma_conv ? ld_conv(cb + D.off_ws, (int64_t)cl * W + jj, cbf) : ld_conv(p.w, (int64_t)c * W + jj, cbf),
                   win[jj], z);
        ys[cl] = z / (1.f + expf(-z));  // SiLU
        for (int jj = 0; jj < W - 1; ++jj) st_conv(page, (int64_t)c * (W - 1) + jj, win[jj + 1], cbf);
      }
      if (tid < G) {
        ys[D.nch + tid] = p.alpha[(int64_t)i * p.Hv + g * G + tid];
        ys[D.nch + G + tid] = p.beta[(int64_t)i * p.Hv + g * G + tid];
      }
      consumer_sync();
      float sq = 0.f, sk = 0.f, sqk = 0.f;
      for (int c = tid; c < DK; c += kConsumers) {
        const float a = ys[c], bk = ys[DK + c];
        sq = fmaf(a, a, sq);
        sk = fmaf(bk, bk, sk);
        sqk = fmaf(a, bk, sqk);
      }
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, m);
      }
      if ((tid & 31) == 0) {
        red[0][tid >> 5] = sq;
        red[1][tid >> 5] = sk;
        red[2][tid >> 5] = sqk;
      }
      consumer_sync();
      sq = sk = sqk = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers / 32; ++w) {
        sq += red[0][w];
        sk += red[1][w];
        sqk += red[2][w];
      }
      const float inv_q = 1.f / sqrtf(sq + 1e-6f);
      const float inv_k = 1.f / sqrtf(sk + 1e-6f);
      kq = sqk * inv_q * inv_k;
#pragma unroll
      for (int jj = 0; jj < Sh::NV; ++jj) {
        const int c0v = (jj * Sh::TPR + lr) * Sh::EPV;
#pragma unroll
        for (int e = 0; e < Sh::EPV; ++e) {
          qreg[jj * Sh::EPV + e] = ys[c0v + e] * inv_q;
          kreg[jj * Sh::EPV + e] = ys[DK + c0v + e] * inv_k;
        }
      }
    }

    // the item's state tiles
    for (int tl = 0; tl < D.TPG; ++tl, ++t) {
      const int stage = t % NS;
      if (consumer_any(!mbar_wait_bounded(&full[stage], (t / NS) & 1, p.wait_limit_ns))) {
        if (tid == 0) report(p.status, LSC_ERR_DEV_TIMEOUT);
        return;
      }
      const int hl = tl / D.TPH, rb = tl % D.TPH;
      const int rows = min(D.TR, dv - rb * D.TR);
      TS *S = reinterpret_cast<TS *>(smem + (int64_t)stage * D.stage_stride);
      float *o = p.out + ((int64_t)i * p.Hv + g * G + hl) * dv + (int64_t)rb * D.TR;
      if (valid) {
        const float a = ys[D.nch + hl], bb = ys[D.nch + G + hl];
        const float *vs = ys + 2 * DK + hl * dv + rb * D.TR;
        const int npass = (rows + Sh::RPP - 1) / Sh::RPP;
        for (int r0 = tid / Sh::TPR; r0 < npass * Sh::RPP; r0 += Sh::RPP) {
          const bool rv = r0 < rows;
          const int r = rv ? r0 : 0;
          float s[Sh::NC];
#pragma unroll
          for (int jj = 0; jj < Sh::NV; ++jj) {
            const uint4 v = warm ? *reinterpret_cast<const uint4 *>(S + (int64_t)r * DK + (jj * Sh::TPR + lr) * Sh::EPV)
                                 : make_uint4(0, 0, 0, 0);
            StateVec<TS>::unpack(v, s + jj * Sh::EPV);
          }
          float u0 = 0.f, u1 = 0.f, w0 = 0.f, w1 = 0.f;
#pragma unroll
          for (int e = 0; e < Sh::NC; e += 2) {
            u0 = fmaf(s[e], kreg[e], u0);
            u1 = fmaf(s[e + 1], kreg[e + 1], u1);
            w0 = fmaf(s[e], qreg[e], w0);
            w1 = fmaf(s[e + 1], qreg[e + 1], w1);
          }
          float u = u0 + u1, wq = w0 + w1;
#pragma unroll
          for (int m = Sh::TPR / 2; m >= 1; m >>= 1) {
            u += __shfl_xor_sync(0xffffffffu, u, m);
            wq += __shfl_xor_sync(0xffffffffu, wq, m);
          }
          const float d = bb * ((rv ? vs[r] : 0.f) - a * u);
          if (rv) {
#pragma unroll
            for (int e = 0; e < Sh::NC; ++e) s[e] = fmaf(a, s[e], d * kreg[e]);
#pragma unroll
            for (int jj = 0; jj < Sh::NV; ++jj)
              *reinterpret_cast<uint4 *>(S + (int64_t)r * DK + (jj * Sh::TPR + lr) * Sh::EPV) =
                  StateVec<TS>::pack(s + jj * Sh::EPV);
            if (lr == 0) o[r] = fmaf(a, wq, d * kq);
          }
        }
      } else {
        for (int r = tid; r < rows; r += kConsumers) o[r] = 0.f;
      }
      fence_proxy_async_smem();
      consumer_sync();
      if (tid == 0) mbar_arrive(&empty[stage]);
    }
  }
}

template <int DK, typename TS>
int launch_decode_t(const DecodeParams &p0, cudaStream_t stream) {
  DecodeParams p = p0;
  const int esc = p.conv_bf16 ? 2 : 4;
  static int optin = 0;  // per process: the opt-in shared-memory limit of a block
  if (!optin) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_CUDA;
    }
  }
  const DecodeGeom probe(DK, (int)sizeof(TS), p.dv, p.group, p.conv_width, esc, 0);
  const int64_t fixed = probe.total + 1024;  // conv, y and item buffers, static shared memory
  int64_t ns = (optin - fixed) / probe.stage_stride;
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return LSC_ERR_UNSUPPORTED;
  p.stages = (int)ns;
  const DecodeGeom D(DK, (int)sizeof(TS), p.dv, p.group, p.conv_width, esc, p.stages);
  static int configured = 0;  // per instantiation
  if (configured < D.total) {
    if (cudaFuncSetAttribute(decode_kernel<DK, TS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)D.total) !=
        cudaSuccess) {
      cudaGetLastError();
      return LSC_ERR_UNSUPPORTED;
    }
    configured = (int)D.total;
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
    decode_kernel<DK, TS><<<grid, kDecodeBlock, (size_t)D.total, stream>>>(q);
    if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  }
  return LSC_OK;
}

// ---------------------------------------------------------------------------
// Token-by-token recurrence.  Grid (Hv, n_seq), one CTA per (sequence, v head);
// row r of the head's state lives in the registers of TPR threads (CPT columns
// each) for the whole sequence.  Tokens are staged in shared memory TT at a
// time; k . q of each token is computed once per tile.
constexpr int kTileTokens = 16;

template <int DK, typename TS>
__global__ void __launch_bounds__(512, 1) recurrent_kernel(const __grid_constant__ RecurrentParams p) {
  constexpr int CPT = DK < 32 ? DK : 32;
  constexpr int TPR = DK / CPT;
  constexpr int NV4 = CPT / 4;
  constexpr int TT = kTileTokens;
  __shared__ __align__(16) float sq[TT][DK];
  __shared__ __align__(16) float sk[TT][DK];
  __shared__ float sv[TT][kMaxDv];
  __shared__ float sa[TT], sb[TT], skq[TT];

  const int tid = threadIdx.x, nthr = blockDim.x;
  const int h = blockIdx.x, i = blockIdx.y;
  const int g = h / p.group;
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
  const int dv = p.dv;
  const int r = tid / TPR, lr = tid % TPR;
  const bool rv = r < dv;

  if (!valid) {  // uniform over the CTA
    for (int64_t e = tid; e < (int64_t)(t1 - t0) * dv; e += nthr) {
      const int64_t t = t0 + e / dv;
      p.out[(t * p.Hv + h) * dv + e % dv] = 0.f;
    }
    return;
  }

  TS *Srow = (TS *)(p.layer + (int64_t)slot * p.page + p.ssm_off) + ((int64_t)h * dv + (rv ? r : 0)) * DK;
  float S[CPT];
#pragma unroll
  for (int j = 0; j < NV4; ++j) {
    const int c0 = (j * TPR + lr) * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = 0.f;
      if (warm && rv) {
        if constexpr (sizeof(TS) == 4) v = ((const float *)Srow)[c0 + e];
        else v = bf16_bits_to_float(((const uint16_t *)Srow)[c0 + e]);
      }
      S[j * 4 + e] = v;
    }
  }

  const int nwarps = (nthr + 31) >> 5, warp = tid >> 5, lane = tid & 31;
  for (int tb = t0; tb < t1; tb += TT) {
    const int nt = t1 - tb < TT ? t1 - tb : TT;
    __syncthreads();
    for (int e = tid; e < nt * (DK / 4); e += nthr) {
      const int tt = e / (DK / 4), c4 = e % (DK / 4);
      const int64_t src = ((int64_t)(tb + tt) * p.Hk + g) * DK + c4 * 4;
      *(float4 *)&sq[tt][c4 * 4] = *(const float4 *)(p.q + src);
      *(float4 *)&sk[tt][c4 * 4] = *(const float4 *)(p.k + src);
    }
    for (int e = tid; e < nt * dv; e += nthr) {
      const int tt = e / dv, c = e % dv;
      sv[tt][c] = p.v[((int64_t)(tb + tt) * p.Hv + h) * dv + c];
    }
    if (tid < nt) {
      sa[tid] = p.alpha[(int64_t)(tb + tid) * p.Hv + h];
      sb[tid] = p.beta[(int64_t)(tb + tid) * p.Hv + h];
    }
    __syncthreads();
    for (int tt = warp; tt < nt; tt += nwarps) {
      float acc = 0.f;
      for (int c = lane; c < DK; c += 32) acc = fmaf(sq[tt][c], sk[tt][c], acc);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
      if (lane == 0) skq[tt] = acc;
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      // four partial sums per dot product keep the FMA chains short
      float u4[4] = {0.f, 0.f, 0.f, 0.f}, w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < NV4; ++j) {
        const int c0 = (j * TPR + lr) * 4;
        const float4 k4 = *(const float4 *)&sk[tt][c0];
        const float4 q4 = *(const float4 *)&sq[tt][c0];
        u4[0] = fmaf(S[j * 4], k4.x, u4[0]); u4[1] = fmaf(S[j * 4 + 1], k4.y, u4[1]);
        u4[2] = fmaf(S[j * 4 + 2], k4.z, u4[2]); u4[3] = fmaf(S[j * 4 + 3], k4.w, u4[3]);
        w4[0] = fmaf(S[j * 4], q4.x, w4[0]); w4[1] = fmaf(S[j * 4 + 1], q4.y, w4[1]);
        w4[2] = fmaf(S[j * 4 + 2], q4.z, w4[2]); w4[3] = fmaf(S[j * 4 + 3], q4.w, w4[3]);
      }
      float u = (u4[0] + u4[1]) + (u4[2] + u4[3]);
      float wq = (w4[0] + w4[1]) + (w4[2] + w4[3]);
#pragma unroll
      for (int m = TPR / 2; m >= 1; m >>= 1) {
        u += __shfl_xor_sync(0xffffffffu, u, m);
        wq += __shfl_xor_sync(0xffffffffu, wq, m);
      }
      const float a = sa[tt], b = sb[tt];
      const float vr = rv ? sv[tt][r] : 0.f;
      const float d = b * (vr - a * u);
#pragma unroll
      for (int j = 0; j < NV4; ++j) {
        const int c0 = (j * TPR + lr) * 4;
        const float4 k4 = *(const float4 *)&sk[tt][c0];
        S[j * 4] = fmaf(a, S[j * 4], d * k4.x);
        S[j * 4 + 1] = fmaf(a, S[j * 4 + 1], d * k4.y);
        S[j * 4 + 2] = fmaf(a, S[j * 4 + 2], d * k4.z);
        S[j * 4 + 3] = fmaf(a, S[j * 4 + 3], d * k4.w);
      }
      if (rv && lr == 0) p.out[((int64_t)(tb + tt) * p.Hv + h) * dv + r] = fmaf(a, wq, d * skq[tt]);
    }
  }

  if (rv) {
#pragma unroll
    for (int j = 0; j < NV4; ++j) {
      const int c0 = (j * TPR + lr) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (sizeof(TS) == 4) ((float *)Srow)[c0 + e] = S[j * 4 + e];
        else ((uint16_t *)Srow)[c0 + e] = float_to_bf16_bits(S[j * 4 + e]);
      }
    }
  }
}

template <int DK, typename TS>
int launch_recurrent_t(const RecurrentParams &p, cudaStream_t s) {
  constexpr int CPT = DK < 32 ? DK : 32;
  constexpr int TPR = DK / CPT;
  int threads = (p.dv * TPR + 31) / 32 * 32;
  if (threads > 512) return LSC_ERR_UNSUPPORTED;
  recurrent_kernel<DK, TS><<<dim3(p.Hv, p.n_seq, 1), threads, 0, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return LSC_ERR_CUDA;
  return LSC_OK;
}

}  // namespace

int launch_decode(const DecodeParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (p.dv > kMaxDv || p.conv_width > kMaxTaps || p.group > 8) return LSC_ERR_UNSUPPORTED;
  const bool bf = ssm_dtype == LSC_BF16;
  switch (dk) {
    case 16: return bf ? launch_decode_t<16, __nv_bfloat16>(p, s) : launch_decode_t<16, float>(p, s);
    case 32: return bf ? launch_decode_t<32, __nv_bfloat16>(p, s) : launch_decode_t<32, float>(p, s);
    case 64: return bf ? launch_decode_t<64, __nv_bfloat16>(p, s) : launch_decode_t<64, float>(p, s);
    case 128: return bf ? launch_decode_t<128, __nv_bfloat16>(p, s) : launch_decode_t<128, float>(p, s);
    default: return LSC_ERR_UNSUPPORTED;
  }
}

int launch_recurrent(const RecurrentParams &p, int dk, int ssm_dtype, cudaStream_t s) {
  if (p.dv > kMaxDv) return LSC_ERR_UNSUPPORTED;
  const bool bf = ssm_dtype == LSC_BF16;
  switch (dk) {
    case 16: return bf ? launch_recurrent_t<16, __nv_bfloat16>(p, s) : launch_recurrent_t<16, float>(p, s);
    case 32: return bf ? launch_recurrent_t<32, __nv_bfloat16>(p, s) : launch_recurrent_t<32, float>(p, s);
    case 64: return bf ? launch_recurrent_t<64, __nv_bfloat16>(p, s) : launch_recurrent_t<64, float>(p, s);
    case 128: return bf ? launch_recurrent_t<128, __nv_bfloat16>(p, s) : launch_recurrent_t<128, float>(p, s);
    default: return LSC_ERR_UNSUPPORTED;
  }
}

}  // namespace lsc
