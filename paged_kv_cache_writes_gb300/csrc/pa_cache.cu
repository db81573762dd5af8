// pa_cache.cu -- cache write (reshape_and_cache) and block copy (copy-on-write).
//
// Both are pure data movement, bound by HBM latency at the batch sizes of a
// decode step: each thread moves one 16-byte vector (8 elements), so a warp
// moves 512 contiguous bytes of one token row.
//
// Cache write: "Inside vLLM Architecture", section "The Block Table Mapping
// Subsystem" (allocate_slot's block = slot / block_size, offset = slot %
// block_size).  fp8 store: "High-Throughput LLM Serving with vLLM &
// PagedAttention", section "4. Production vLLM Docker Deployment with FP8
// Quantization" (--kv-cache-dtype fp8); stored code = e4m3(fp32(x) / scale),
// IEEE division, round to nearest even, saturating.
// Block copy: same page, section "2. Virtual Memory Paging Applied to GPUs"
// (copy-on-write when branches diverge).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

// One thread per 16-byte vector of input: index = ((t * 2 + side) * Hkv + h) * (D/8) + j.
template <typename In, bool kFp8>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const In *__restrict__ k, const In *__restrict__ v, int64_t num_tokens, int64_t token_stride,
    const int64_t *__restrict__ slot_mapping, void *__restrict__ k_cache, void *__restrict__ v_cache,
    int64_t num_slots, int32_t block_size, int32_t num_kv_heads, int32_t head_dim, float k_scale,
    float v_scale, const float *__restrict__ k_hs, const float *__restrict__ v_hs, int32_t *err) {
  const int32_t vec_per_head = head_dim >> 3;
  const int64_t per_token = 2ll * num_kv_heads * vec_per_head;
  const int64_t total = num_tokens * per_token;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / per_token;
    int64_t rem = idx - t * per_token;
    const int side = rem >= per_token / 2;
    rem -= side * (per_token / 2);
    const int32_t h = (int32_t)(rem / vec_per_head);
    const int32_t j = (int32_t)(rem - (int64_t)h * vec_per_head);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      record_error(err, PA_ERR_DEVICE_CHECK);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot - blk * block_size;
    const In *src = (side ? v : k) + t * token_stride + (int64_t)h * head_dim + j * 8;
    const int64_t dst_elem = ((blk * num_kv_heads + h) * block_size + off) * head_dim + j * 8;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(src));
    if constexpr (!kFp8) {
      In *dst = static_cast<In *>(side ? v_cache : k_cache) + dst_elem;
      *reinterpret_cast<uint4 *>(dst) = x;
    } else {
      const float s = k_hs ? __ldg((side ? v_hs : k_hs) + h) : side ? v_scale : k_scale;   // per head, or per pool
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t out[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2(w[i], In{});
        const float2 qv = make_float2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s));
        const uint32_t pair = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
        if (i & 1) out[i >> 1] |= pair << 16;
        else out[i >> 1] = pair;
      }
      uint8_t *dst = static_cast<uint8_t *>(side ? v_cache : k_cache) + dst_elem;
      *reinterpret_cast<uint2 *>(dst) = make_uint2(out[0], out[1]);
    }
  }
}

// grid.x = pair, grid.y = 0 (K) / 1 (V); each CTA copies one block of one pool.
__global__ void __launch_bounds__(256) copy_blocks_kernel(char *__restrict__ k_cache,
                                                          char *__restrict__ v_cache,
                                                          const int32_t *__restrict__ pairs,
                                                          int64_t num_blocks, int64_t block_bytes,
                                                          int32_t *err) {
  const int32_t src = __ldg(pairs + 2 * blockIdx.x), dst = __ldg(pairs + 2 * blockIdx.x + 1);
  if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) record_error(err, PA_ERR_DEVICE_CHECK);
    return;
  }
  char *base = blockIdx.y ? v_cache : k_cache;
  const uint4 *s = reinterpret_cast<const uint4 *>(base + src * block_bytes);
  uint4 *d = reinterpret_cast<uint4 *>(base + dst * block_bytes);
  const int64_t n = block_bytes >> 4;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = __ldg(s + i);
}

cudaError_t launch_reshape_and_cache(const void *k, const void *v, pa_dtype in_dtype,
                                     int64_t num_tokens, int64_t token_stride,
                                     const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                     const pa_kv_cache &c, int32_t *err, cudaStream_t stream) {
  const int64_t total = num_tokens * 2 * c.num_kv_heads * (c.head_dim / 8);
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  const unsigned grid = (unsigned)(blocks < 65535 * 8 ? blocks : 65535 * 8);
  const int64_t num_slots = c.num_blocks * c.block_size;
  const bool fp8 = c.kv_dtype == PA_FP8_E4M3;
#define PA_RAC(T, F)                                                                         \
  reshape_and_cache_kernel<T, F><<<grid, threads, 0, stream>>>(                              \
      static_cast<const T *>(k), static_cast<const T *>(v), num_tokens, token_stride,        \
      slot_mapping, k_cache, v_cache, num_slots, c.block_size, c.num_kv_heads, c.head_dim,   \
      c.k_scale, c.v_scale, c.k_head_scales, c.v_head_scales, err)
  if (in_dtype == PA_BF16) {
    if (fp8) PA_RAC(__nv_bfloat16, true);
    else PA_RAC(__nv_bfloat16, false);
  } else {
    if (fp8) PA_RAC(__half, true);
    else PA_RAC(__half, false);
  }
#undef PA_RAC
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const pa_kv_cache &c,
                               const int32_t *pairs, int32_t num_pairs, int32_t *err,
                               cudaStream_t stream) {
  const int64_t block_bytes =
      (int64_t)c.num_kv_heads * c.block_size * c.head_dim * dtype_bytes(c.kv_dtype);
  copy_blocks_kernel<<<dim3(num_pairs, 2), 256, 0, stream>>>(
      static_cast<char *>(k_cache), static_cast<char *>(v_cache), pairs, c.num_blocks, block_bytes,
      err);
  return cudaGetLastError();
}

}  // namespace pa
