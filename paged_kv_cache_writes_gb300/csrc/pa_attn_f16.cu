// pa_attn_f16.cu -- paged attention instantiations for a f16 cache, f16 queries: the
// persistent decode kernel and the CUDA-core prefill-row kernel.  One
// translation unit per dtype pair so the library compiles in parallel.
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_attention_f16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                  cudaStream_t s) {
  return launch_attention<__half, __half>(p, m, head_dim, rows, s);
}
cudaError_t launch_decode_f16(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                               cudaStream_t s) {
  return launch_decode<__half, __half>(p, hpc, m, head_dim, s);
}
}  // namespace pa
