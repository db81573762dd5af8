// pa_decode_tc_bf16.cu -- tensor-core decode instantiations for a bf16 cache.
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_bf16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                  cudaStream_t s) {
  return launch_decode_tc<__nv_bfloat16, __nv_bfloat16>(p, gqa, head_dim, m, s);
}
}  // namespace pa
