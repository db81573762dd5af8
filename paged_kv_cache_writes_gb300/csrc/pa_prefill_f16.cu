// pa_prefill_f16.cu -- tensor-core chunked-prefill instantiations for an f16
// cache with f16 queries.
#include "pa_prefill_tc.cuh"

namespace pa {
cudaError_t launch_prefill_tc_f16(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                  cudaStream_t s) {
  return launch_prefill_tc<__half, __half>(p, m, gqa, num_chunks, s);
}
}  // namespace pa
