// pa_attn_bf16.cu -- paged attention instantiations for a bf16 cache, bf16 queries: the
// persistent decode kernel and the CUDA-core prefill-row kernel.  One
// translation unit per dtype pair so the library compiles in parallel.
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_attention_bf16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                  cudaStream_t s) {
  return launch_attention<__nv_bfloat16, __nv_bfloat16>(p, m, head_dim, rows, s);
}
cudaError_t launch_decode_bf16(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                               cudaStream_t s) {
  return launch_decode<__nv_bfloat16, __nv_bfloat16>(p, hpc, m, head_dim, s);
}
}  // namespace pa
