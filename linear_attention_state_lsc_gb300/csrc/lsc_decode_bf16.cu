// lsc_decode_bf16.cu -- fused GDN decode instantiations for bf16 ssm state.
#include "lsc_decode.cuh"

namespace lsc {
int launch_decode_bf16(const DecodeParams &p, int dk, cudaStream_t s) { return launch_decode_ts<__nv_bfloat16>(p, dk, s); }
}  // namespace lsc
