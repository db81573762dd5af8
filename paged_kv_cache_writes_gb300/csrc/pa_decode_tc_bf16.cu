// pa_decode_tc_bf16.cu -- tensor-core decode instantiations for a bf16 cache.
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_bf16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                  cudaStream_t s) {
  if (!decode_tc_exact_group(head_dim, gqa)) return launch_decode_tc_pad_bf16(p, gqa, head_dim, m, s);
  return launch_decode_tc<__nv_bfloat16, __nv_bfloat16, false>(p, gqa, head_dim, m, s);
}
}  // namespace pa
