// pa_attn_f16.cu -- paged attention instantiations for a f16 cache, f16 queries.
// One translation unit per dtype pair so the library compiles in parallel.
#include "pa_attention.cuh"

namespace pa {
cudaError_t launch_attention_f16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                cudaStream_t s) {
  return launch_attention<__half, __half>(p, m, head_dim, rows, s);
}
}  // namespace pa
