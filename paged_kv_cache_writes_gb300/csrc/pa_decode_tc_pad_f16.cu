// pa_decode_tc_pad_f16.cu -- tensor-core decode instantiations for an f16
// cache and query groups other than 4, 8 and 16 heads per KV head (run with
// padding rows), in a translation unit of their own for a parallel build.
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_pad_f16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                     cudaStream_t s) {
  return launch_decode_tc<__half, __half, true>(p, gqa, head_dim, m, s);
}
}  // namespace pa
