// pa_attn_bf16.cu -- paged attention instantiations for a bf16 cache, bf16 queries.
// One translation unit per dtype pair so the library compiles in parallel.
#include "pa_attention.cuh"

namespace pa {
cudaError_t launch_attention_bf16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                 cudaStream_t s) {
  return launch_attention<__nv_bfloat16, __nv_bfloat16>(p, m, head_dim, rows, s);
}
}  // namespace pa
