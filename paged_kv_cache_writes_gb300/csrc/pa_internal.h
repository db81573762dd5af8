// pa_internal.h -- host-side interface between the C ABI (pa_api.cu) and the
// kernel launchers.  Not installed; not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pa.h"

namespace pa {

inline int dtype_bytes(pa_dtype t) { return t == PA_FP8_E4M3 ? 1 : 2; }

// Raise kernel Kern's dynamic shared-memory limit to `bytes`, once per device
// (the attribute belongs to the function on the current device; setting it on
// every launch would cost a driver call per launch).
template <auto Kern>
inline cudaError_t ensure_smem_limit(int bytes) {
  static std::atomic<uint64_t> done{0};  // bit d: set on device d (devices 0..63; others every call)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Number of SMs of the current device (queried once per device).
inline cudaError_t current_sm_count(int *sms) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *sms = v;
      return cudaSuccess;
    }
  }
  int v = 0;
  if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
  *sms = v;
  return cudaSuccess;
}

constexpr int kDefaultPartition = 512;   // split-KV partition, tokens (also the largest used)
constexpr int kMaxPartitions = 4096;     // per sequence (item encoding: 12 bits)
constexpr int kMaxDecodeRows = 1 << 19;  // sequences per call (item encoding: row << 12)

// Decode / CUDA-core prefill parameters shared by every instantiation.
struct AttnParams {
  const void *q;              // [rows][Hq][D]
  void *out;                  // [rows][Hq][D]
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  // decode: one row per sequence, row i has seq_lens[i] tokens
  const int32_t *seq_lens;
  // prefill (cu_q_lens != nullptr): row (c, r) has q_start[c] + r + 1 tokens
  const int32_t *cu_q_lens;
  const int32_t *q_start;
  int32_t max_q_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t heads_per_cta;      // query heads one CTA serves (share one KV read)
  int32_t block_size;
  int64_t num_blocks;
  int32_t partition_size;     // tokens per split-KV partition (multiple of 32)
  int32_t max_partitions;     // grid.z
  float q_mult;               // softmax scale * log2(e) (* k_scale for fp8)
  float out_mult;             // v_scale for fp8, else 1
  const float *k_hs;          // fp8, optional: [Hkv] per-head scales multiplying q_mult / out_mult
  const float *v_hs;
  int32_t out_f32;            // 1: out is fp32; 0: out has the query dtype
  // split-KV workspace (null when max_partitions == 1)
  float *ws_acc;              // [rows][Hq][max_partitions][D]
  float2 *ws_ml;              // [rows][Hq][max_partitions] (max, sum) in log2 units
  int32_t *ws_count;          // [rows][Hq] arrival counters (self-resetting)
  int32_t *err;               // device error word
};

// Decode workspace: header | item list | split-KV partials (acc, max/sum) | counters.
struct WorkspaceLayout {
  size_t hdr_off, items_off, acc_off, ml_off, cnt_off, jobs_off, total;
};
WorkspaceLayout decode_workspace_layout(int64_t rows, int64_t num_q_heads, int64_t head_dim,
                                        int64_t max_partitions);

cudaError_t launch_reshape_and_cache(const void *k, const void *v, pa_dtype in_dtype,
                                     int64_t num_tokens, int64_t token_stride,
                                     const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                     const pa_kv_cache &c, int32_t *err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const pa_kv_cache &c,
                               const int32_t *pairs, int32_t num_pairs, int32_t *err,
                               cudaStream_t stream);

// Tensor maps over one pool viewed as a 2D array [num_blocks*Hkv*bs rows][D].
struct PoolMaps {
  CUtensorMap k, v;
};
// The decode kernel reads 256-byte rows as one 3D box of two 128-byte panels.

struct DecodeParams;     // pa_decode.cuh
struct DecodeTcParams;   // pa_decode_tc.cuh
struct PrefillTcParams;  // pa_prefill_tc.cuh

// Launch the CUDA-core prefill-row kernel / the persistent decode for one (kv dtype, q dtype).
cudaError_t launch_attention_bf16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                  cudaStream_t s);
cudaError_t launch_attention_f16(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                                 cudaStream_t s);
cudaError_t launch_attention_fp8_bf16q(const AttnParams &p, const PoolMaps &m, int head_dim,
                                       int rows, cudaStream_t s);
cudaError_t launch_attention_fp8_f16q(const AttnParams &p, const PoolMaps &m, int head_dim,
                                      int rows, cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                               cudaStream_t s);
cudaError_t launch_decode_f16(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                              cudaStream_t s);
cudaError_t launch_decode_fp8_bf16q(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                                    cudaStream_t s);
cudaError_t launch_decode_fp8_f16q(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                                   cudaStream_t s);

// Tensor-core decode: head_dim 128 with gqa = Hq / Hkv in 1..16, or head_dim 64 with
// gqa in 1..8 (a group runs padded to 4, 8 or 16 query rows); one query head per KV
// head with a 16-bit cache stays on the CUDA-core kernel, measured faster there
// (128 sequences: 0.191 against 0.198 ms with head_dim 128, 0.115 against 0.137 with 64).
// A group the tensor-core decode runs without padding rows.
constexpr bool decode_tc_exact_group(int head_dim, int gqa) {
  return gqa == 4 || gqa == 8 || (gqa == 16 && head_dim == 128);
}
constexpr bool decode_tc_supported(int head_dim, int gqa, pa_dtype kv) {
  return ((head_dim == 128 && gqa >= 1 && gqa <= 16) || (head_dim == 64 && gqa >= 1 && gqa <= 8)) &&
         (gqa >= 2 || kv == PA_FP8_E4M3);
}
// exact groups here; the other groups by the _pad launchers (their own translation units)
cudaError_t launch_decode_tc_bf16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m, cudaStream_t s);
cudaError_t launch_decode_tc_pad_bf16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                      cudaStream_t s);
cudaError_t launch_decode_tc_pad_f16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                     cudaStream_t s);
cudaError_t launch_decode_tc_pad_fp8_bf16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                           cudaStream_t s);
cudaError_t launch_decode_tc_pad_fp8_f16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                          cudaStream_t s);
cudaError_t launch_decode_tc_f16(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m, cudaStream_t s);
cudaError_t launch_decode_tc_fp8_bf16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                       cudaStream_t s);
cudaError_t launch_decode_tc_fp8_f16q(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m,
                                      cudaStream_t s);

// One launch for a prefill chunk batch and a decode batch (pa_mixed_tc.cuh):
// both on the tensor cores, head_dim 128, 4 or 8 query heads per KV head.
constexpr bool mixed_tc_supported(int head_dim, int gqa) { return head_dim == 128 && (gqa == 4 || gqa == 8); }
cudaError_t launch_mixed_tc_bf16(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p, int num_chunks,
                                 int gqa, cudaStream_t s);
cudaError_t launch_mixed_tc_f16(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p, int num_chunks,
                                int gqa, cudaStream_t s);
cudaError_t launch_mixed_tc_fp8_bf16q(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                      int num_chunks, int gqa, cudaStream_t s);
cudaError_t launch_mixed_tc_fp8_f16q(const DecodeTcParams &d, const PoolMaps &m, const PrefillTcParams &p,
                                     int num_chunks, int gqa, cudaStream_t s);

// Tensor-core chunked prefill (head_dim 128; gqa = Hq / Hkv in {1, 2, 4, 8, 16}).
constexpr bool prefill_tc_supported(int head_dim, int gqa) {
  return head_dim == 128 && (gqa == 1 || gqa == 2 || gqa == 4 || gqa == 8 || gqa == 16);
}
cudaError_t launch_prefill_tc_bf16(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                   cudaStream_t s);
cudaError_t launch_prefill_tc_f16(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                  cudaStream_t s);
cudaError_t launch_prefill_tc_fp8_bf16q(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                        cudaStream_t s);
cudaError_t launch_prefill_tc_fp8_f16q(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks,
                                       cudaStream_t s);

}  // namespace pa
