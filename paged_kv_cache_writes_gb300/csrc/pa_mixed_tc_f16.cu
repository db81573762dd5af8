// pa_mixed_tc_f16.cu -- one-launch prefill + decode instantiations for an f16 cache.
#include "pa_mixed_tc.cuh"

namespace pa {
cudaError_t launch_mixed_tc_f16(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                 int num_chunks, int gqa, cudaStream_t s) {
  return launch_mixed_tc<__half, __half>(d, m, p, num_chunks, gqa, s);
}
}  // namespace pa
