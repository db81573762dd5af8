// pa_attn_fp8_bf16q.cu -- paged attention instantiations for a fp8-e4m3 cache, bf16 queries: the
// persistent decode kernel and the CUDA-core prefill-row kernel.  One
// translation unit per dtype pair so the library compiles in parallel.
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_attention_fp8_bf16q(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                  cudaStream_t s) {
  return launch_attention<uint8_t, __nv_bfloat16>(p, m, head_dim, rows, s);
}
cudaError_t launch_decode_fp8_bf16q(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                               cudaStream_t s) {
  return launch_decode<uint8_t, __nv_bfloat16>(p, hpc, m, head_dim, s);
}
}  // namespace pa
