// lsc_decode_f32.cu -- fused GDN decode instantiations for f32 ssm state.
#include "lsc_decode.cuh"

namespace lsc {
int launch_decode_f32(const DecodeParams &p, int dk, cudaStream_t s) { return launch_decode_ts<float>(p, dk, s); }
}  // namespace lsc
