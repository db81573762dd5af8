// pa_decode_tc_fp8.cu -- tensor-core decode instantiations for an fp8-e4m3
// cache, with bf16 or f16 queries (the codes enter kind::f8f6f4 MMAs as stored).
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_fp8_bf16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                       cudaStream_t s) {
  if (!decode_tc_exact_group(head_dim, gqa)) return launch_decode_tc_pad_fp8_bf16q(p, gqa, head_dim, m, s);
  return launch_decode_tc<uint8_t, __nv_bfloat16, false>(p, gqa, head_dim, m, s);
}
cudaError_t launch_decode_tc_fp8_f16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                      cudaStream_t s) {
  if (!decode_tc_exact_group(head_dim, gqa)) return launch_decode_tc_pad_fp8_f16q(p, gqa, head_dim, m, s);
  return launch_decode_tc<uint8_t, __half, false>(p, gqa, head_dim, m, s);
}
}  // namespace pa
