// pa_decode_tc_f16.cu -- tensor-core decode instantiations for an f16 cache.
#include "pa_decode_tc.cuh"

namespace pa {
cudaError_t launch_decode_tc_f16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                 cudaStream_t s) {
  if (!decode_tc_exact_group(head_dim, gqa)) return launch_decode_tc_pad_f16(p, gqa, head_dim, m, s);
  return launch_decode_tc<__half, __half, false>(p, gqa, head_dim, m, s);
}
}  // namespace pa
