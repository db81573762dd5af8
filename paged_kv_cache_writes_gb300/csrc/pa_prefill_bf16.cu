// pa_prefill_bf16.cu -- tensor-core chunked-prefill instantiations for a bf16
// cache with bf16 queries (one translation unit per cache dtype so the
// library compiles in parallel).
#include "pa_prefill_tc.cuh"

namespace pa {
cudaError_t launch_prefill_tc_bf16(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                   cudaStream_t s) {
  return launch_prefill_tc<__nv_bfloat16, __nv_bfloat16>(p, m, gqa, num_chunks, s);
}
}  // namespace pa
