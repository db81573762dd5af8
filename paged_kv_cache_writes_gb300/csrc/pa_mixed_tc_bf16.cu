// pa_mixed_tc_bf16.cu -- one-launch prefill + decode instantiations for a bf16 cache.
#include "pa_mixed_tc.cuh"

namespace pa {
cudaError_t launch_mixed_tc_bf16(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                 int num_chunks, int gqa, cudaStream_t s) {
  return launch_mixed_tc<__nv_bfloat16, __nv_bfloat16>(d, m, p, num_chunks, gqa, s);
}
}  // namespace pa
