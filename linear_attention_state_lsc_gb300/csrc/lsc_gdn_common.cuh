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

}  // namespace lsc
