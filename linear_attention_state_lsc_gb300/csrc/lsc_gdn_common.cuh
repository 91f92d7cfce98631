// lsc_gdn_common.cuh -- device helpers shared by the GDN kernels of liblsc.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "lsc_internal.h"
#include "lsc_ptx.h"

namespace lsc {

constexpr int kMaxDv = 128;   // largest supported head_v_dim
constexpr int kMaxTaps = 8;   // largest supported conv width

__device__ __forceinline__ void report(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// Element access at a compile-time dtype (float or bf16), values as float.
template <typename T> struct Elem;
template <> struct Elem<float> {
  __device__ __forceinline__ static float ld(const void *base, int64_t i) { return ((const float *)base)[i]; }
  __device__ __forceinline__ static void st(void *base, int64_t i, float v) { ((float *)base)[i] = v; }
};
template <> struct Elem<__nv_bfloat16> {
  __device__ __forceinline__ static float ld(const void *base, int64_t i) {
    return bf16_bits_to_float(((const uint16_t *)base)[i]);
  }
  __device__ __forceinline__ static void st(void *base, int64_t i, float v) {
    ((uint16_t *)base)[i] = float_to_bf16_bits(v);
  }
};

// Pairs of floats in one 64-bit register (low half = first element) for the
// packed f32x2 arithmetic of sm_100 and later: one instruction does two
// independent, individually rounded fp32 operations.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The sequence a CTA of a per-sequence grid takes.  With at most kRankedSeqs
// sequences, the CTA with blockIdx.y = b takes the sequence of rank b by
// length (longest first, ties by index), so that long sequences do not start
// last; otherwise sequence b.  Every thread of the CTA calls it.
constexpr int kRankedSeqs = 256;
__device__ __forceinline__ int ranked_sequence(const int32_t *cu, int n_seq, int32_t *s_len, int32_t *s_seq) {
  if (n_seq > kRankedSeqs) return blockIdx.y;
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) s_len[s] = cu[s + 1] - cu[s];
  __syncthreads();
  for (int s = threadIdx.x; s < n_seq; s += blockDim.x) {
    const int ls = s_len[s];
    int rank = 0;
    for (int j = 0; j < n_seq; ++j) rank += (s_len[j] > ls) || (s_len[j] == ls && j < s);
    if (rank == (int)blockIdx.y) *s_seq = s;
  }
  __syncthreads();
  return *s_seq;
}

// 16-byte vectors of state elements <-> float pairs (EPV / 2 of them).
template <typename TS> struct StatePairs;
template <> struct StatePairs<float> {
  static constexpr int N = 2;
  __device__ __forceinline__ static void unpack(const uint4 &v, uint64_t *f) {
    f[0] = f2_pack(__uint_as_float(v.x), __uint_as_float(v.y));
    f[1] = f2_pack(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ __forceinline__ static uint4 pack(const uint64_t *f) {
    float a, b, c, d;
    f2_unpack(f[0], a, b);
    f2_unpack(f[1], c, d);
    return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c), __float_as_uint(d));
  }
};
template <> struct StatePairs<__nv_bfloat16> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4 &v, uint64_t *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) f[k] = f2_pack(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
  }
  __device__ __forceinline__ static uint4 pack(const uint64_t *f) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float lo, hi;
      f2_unpack(f[k], lo, hi);
      __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // .x = low half
      w[k] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

}  // namespace lsc
