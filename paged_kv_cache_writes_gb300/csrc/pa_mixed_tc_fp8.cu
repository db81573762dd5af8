// pa_mixed_tc_fp8.cu -- one-launch prefill + decode instantiations for an
// fp8-e4m3 cache, with bf16 or f16 queries.
#include "pa_mixed_tc.cuh"

namespace pa {
cudaError_t launch_mixed_tc_fp8_bf16q(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                 int num_chunks, int gqa, cudaStream_t s) {
  return launch_mixed_tc<uint8_t, __nv_bfloat16>(d, m, p, num_chunks, gqa, s);
}
cudaError_t launch_mixed_tc_fp8_f16q(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                 int num_chunks, int gqa, cudaStream_t s) {
  return launch_mixed_tc<uint8_t, __half>(d, m, p, num_chunks, gqa, s);
}
}  // namespace pa
