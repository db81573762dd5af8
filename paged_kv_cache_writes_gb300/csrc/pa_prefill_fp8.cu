// pa_prefill_fp8.cu -- tensor-core chunked-prefill instantiations for an
// fp8-e4m3 cache, with bf16 or f16 queries (the codes are widened to the
// query type in shared memory).
#include "pa_prefill_tc.cuh"

namespace pa {
cudaError_t launch_prefill_tc_fp8_bf16q(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                        cudaStream_t s) {
  return launch_prefill_tc<uint8_t, __nv_bfloat16>(p, m, gqa, num_chunks, s);
}
cudaError_t launch_prefill_tc_fp8_f16q(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                       cudaStream_t s) {
  return launch_prefill_tc<uint8_t, __half>(p, m, gqa, num_chunks, s);
}
}  // namespace pa
