// pa_attn_fp8_bf16q.cu -- paged attention instantiations for a fp8-e4m3 cache, bf16 queries.
// One translation unit per dtype pair so the library compiles in parallel.
#include "pa_attention.cuh"

namespace pa {
cudaError_t launch_attention_fp8_bf16q(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                      cudaStream_t s) {
  return launch_attention<uint8_t, __nv_bfloat16>(p, m, head_dim, rows, s);
}
}  // namespace pa
