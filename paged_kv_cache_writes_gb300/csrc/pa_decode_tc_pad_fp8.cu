// pa_decode_tc_pad_fp8.cu -- tensor-core decode instantiations for an
// fp8-e4m3 cache with bf16 or f16 queries and query groups other than 4, 8
// and 16 heads per KV head (run with padding rows), in a translation unit of
// their own for a parallel build.
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_pad_fp8_bf16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                           cudaStream_t s) {
  return launch_decode_tc<uint8_t, __nv_bfloat16, true>(p, gqa, head_dim, m, s);
}
cudaError_t launch_decode_tc_pad_fp8_f16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                          cudaStream_t s) {
  return launch_decode_tc<uint8_t, __half, true>(p, gqa, head_dim, m, s);
}
}  // namespace pa
