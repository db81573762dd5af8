// pa_api.cu -- the extern "C" entry points of libpa declared in include/pa.h.
//
// Host side only: validate arguments, build the TMA tensor maps of the two
// pools, lay out the split-KV workspace, pick the kernel instantiation and
// enqueue it on the caller's stream.  No call allocates memory or
// synchronises (except pa_get_device_error).
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_decode_tc.cuh"
#include "pa_internal.h"
#include "pa_prefill_tc.cuh"

namespace pa {

__device__ int32_t g_device_error = 0;

// One warp waits on an mbarrier nothing completes; the bounded wait records
// PA_ERR_TIMEOUT and the kernel returns.
__global__ void selftest_wait_kernel(int32_t *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  (void)mbar_wait(&bar, 0, err);
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Address of the current device's error word (a host-side name is not a
// device address; the runtime resolves it per device).
int32_t *device_error_word() {
  void *ptr = nullptr;
  return cudaGetSymbolAddress(&ptr, g_device_error) == cudaSuccess ? static_cast<int32_t *>(ptr)
                                                                   : nullptr;
}
size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

pa_status check_cache(const pa_kv_cache *c) {
  if (c == nullptr || c->num_blocks <= 0 || c->num_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (c->block_size != 16 && c->block_size != 32) return PA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (c->kv_dtype != PA_F16 && c->kv_dtype != PA_BF16 && c->kv_dtype != PA_FP8_E4M3)
    return PA_ERR_UNSUPPORTED;
  if (c->kv_dtype == PA_FP8_E4M3 &&
      !(std::isfinite(c->k_scale) && c->k_scale > 0.f && std::isfinite(c->v_scale) &&
        c->v_scale > 0.f))
    return PA_ERR_INVALID_ARG;
  // per-head scales: both or neither, fp8 only
  if ((c->k_head_scales == nullptr) != (c->v_head_scales == nullptr)) return PA_ERR_INVALID_ARG;
  if (c->k_head_scales && (c->kv_dtype != PA_FP8_E4M3 || !aligned(c->k_head_scales, 4) ||
                           !aligned(c->v_head_scales, 4)))
    return PA_ERR_INVALID_ARG;
  // tile rows of the 2D pool view are addressed with int32 TMA coordinates
  if ((double)c->num_blocks * c->num_kv_heads * c->block_size >= 2147483648.0)
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

pa_status check_pools(const void *k_cache, const void *v_cache) {
  if (!k_cache || !v_cache || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

// q dtype must equal the cache dtype, except that an fp8 cache takes f16/bf16 queries.
pa_status check_q_dtype(pa_dtype q, const pa_kv_cache &c) {
  if (q != PA_F16 && q != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (c.kv_dtype != PA_FP8_E4M3 && q != c.kv_dtype) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

int heads_per_cta(int gqa) { return gqa % 8 == 0 ? 8 : gqa % 4 == 0 ? 4 : 1; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// One pool (256-byte rows) as a 4D tensor of 8-row atoms: dims {64 elements,
// 8 rows (256 B apart), 2 panels (128 B apart), atoms (2048 B apart)}; one box
// is a whole cache block of one KV head (block_size / 8 atoms), landing in
// shared memory as [atom][panel][8 rows][128 B] with the 128-byte swizzle.
// A pool of 128-byte rows (16-bit, head_dim 64) is the 3D tensor {64
// elements, 8 rows, atoms (1024 B apart)}, landing as [atom][8 rows][128 B].
bool encode_pool_map_atoms(CUtensorMap *map, const void *base, const pa_kv_cache &c) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  if (c.kv_dtype != PA_FP8_E4M3 && c.head_dim == 64) {
    const CUtensorMapDataType dt =
        c.kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t dims[3] = {64, 8, (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size / 8};
    const cuuint64_t strides[2] = {128, 1024};
    const cuuint32_t box[3] = {64, 8, (cuuint32_t)(c.block_size / 8)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  if (c.head_dim * dtype_bytes(c.kv_dtype) != 256) return false;
  const CUtensorMapDataType dt = c.kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size / 8};
  const cuuint64_t strides[3] = {256, 128, 2048};
  const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(c.block_size / 8)};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return enc(map, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An fp8 pool as a 2D tensor [rows][head_dim codes]; one box is a whole
// cache block of one KV head (block_size rows), with the 128-byte swizzle
// (head_dim 128) or the 64-byte one (head_dim 64).
bool encode_pool_map_fp8_blocks(CUtensorMap *map, const void *base, const pa_kv_cache &c) {
  auto enc = tensor_map_encoder();
  if (!enc || (c.head_dim != 128 && c.head_dim != 64) || c.kv_dtype != PA_FP8_E4M3) return false;
  const cuuint64_t d = (cuuint64_t)c.head_dim;
  const cuuint64_t dims[2] = {d, (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size};
  const cuuint64_t strides[1] = {d};
  const cuuint32_t box[2] = {(cuuint32_t)d, (cuuint32_t)c.block_size};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One pool as a 2D tensor [num_blocks*Hkv*bs rows][head_dim]; box = 16 rows x
// one 128-byte (or 64-byte) panel, swizzled to match the kernels' reads.  With
// `panels3d` and 256-byte rows the pool is viewed as [2 panels][rows][64] and
// one box covers 16 rows of both panels (same shared-memory layout as two
// 2D boxes).
bool encode_pool_map(CUtensorMap *map, const void *base, const pa_kv_cache &c, bool panels3d = false) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int eb = dtype_bytes(c.kv_dtype);
  const int row_bytes = c.head_dim * eb;
  const int panel_bytes = row_bytes < 128 ? row_bytes : 128;
  const cuuint64_t dims[2] = {(cuuint64_t)c.head_dim,
                              (cuuint64_t)c.num_blocks * c.num_kv_heads * c.block_size};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(panel_bytes / eb), 16u};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUtensorMapDataType dt = c.kv_dtype == PA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : c.kv_dtype == PA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw =
      panel_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (panels3d && row_bytes == 2 * panel_bytes) {
    const cuuint64_t dims3[3] = {(cuuint64_t)(panel_bytes / eb), dims[1], 2};
    const cuuint64_t strides3[2] = {(cuuint64_t)row_bytes, (cuuint64_t)panel_bytes};
    const cuuint32_t box3[3] = {(cuuint32_t)(panel_bytes / eb), 16u, 2u};
    const cuuint32_t estr3[3] = {1u, 1u, 1u};
    return enc(map, dt, 3, const_cast<void *>(base), dims3, strides3, box3, estr3,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  return enc(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t dispatch_attention(pa_dtype q_dtype, const pa_kv_cache &c, const AttnParams &p,
                               const PoolMaps &m, int rows, cudaStream_t s) {
  if (c.kv_dtype == PA_BF16) return launch_attention_bf16(p, m, c.head_dim, rows, s);
  if (c.kv_dtype == PA_F16) return launch_attention_f16(p, m, c.head_dim, rows, s);
  if (q_dtype == PA_BF16) return launch_attention_fp8_bf16q(p, m, c.head_dim, rows, s);
  return launch_attention_fp8_f16q(p, m, c.head_dim, rows, s);
}

}  // namespace

WorkspaceLayout decode_workspace_layout(int64_t rows, int64_t num_q_heads, int64_t head_dim,
                                        int64_t max_partitions) {
  WorkspaceLayout w;
  w.hdr_off = 0;
  w.items_off = round256(sizeof(DecodeHeader));
  w.acc_off = w.items_off + round256((size_t)(rows * max_partitions * 4));
  const int64_t partials = max_partitions > 1 ? rows * num_q_heads * max_partitions : 0;
  w.ml_off = w.acc_off + round256((size_t)(partials * head_dim * 4));
  w.cnt_off = w.ml_off + round256((size_t)(partials * 8));
  w.jobs_off = w.cnt_off + round256((size_t)(rows * num_q_heads * 4));
  // merge list of the tensor-core decode (split rows only)
  w.total = w.jobs_off + round256((size_t)(max_partitions > 1 ? rows * num_q_heads * 16 : 0));
  return w;
}

namespace {
std::atomic<int32_t> g_decode_kernel{PA_DECODE_KERNEL_AUTO};  // pa_set_decode_kernel

int effective_partition(int32_t requested) {
  const int ps = requested ? requested : kDefaultPartition;
  return ps < kDefaultPartition ? ps : kDefaultPartition;  // a unit spans at most 32 blocks
}
}  // namespace

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_reshape_and_cache(const void *k, const void *v, pa_dtype in_dtype, int32_t num_tokens,
                               int64_t token_stride, const int64_t *slot_mapping, void *k_cache,
                               void *v_cache, const pa_kv_cache *cache, pa_stream_t stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (in_dtype != PA_F16 && in_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (cache->kv_dtype != PA_FP8_E4M3 && cache->kv_dtype != in_dtype) return PA_ERR_UNSUPPORTED;
  if (token_stride < (int64_t)cache->num_kv_heads * cache->head_dim || token_stride % 8)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  if ((st = check_pools(k_cache, v_cache)) != PA_OK) return st;
  int32_t *err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  return launch_reshape_and_cache(k, v, in_dtype, num_tokens, token_stride, slot_mapping, k_cache,
                                  v_cache, *cache, err, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void *k_cache, void *v_cache, const pa_kv_cache *cache,
                         const int32_t *src_dst_pairs, int32_t num_pairs, pa_stream_t stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!src_dst_pairs || !aligned(src_dst_pairs, 8)) return PA_ERR_INVALID_ARG;
  if ((st = check_pools(k_cache, v_cache)) != PA_OK) return st;
  int32_t *err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  return launch_copy_blocks(k_cache, v_cache, *cache, src_dst_pairs, num_pairs, err,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_seq_len, int32_t partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
      partition_size < 0 || num_q_heads % num_kv_heads)
    return 0;
  if (partition_size % 32 || num_seqs > kMaxDecodeRows) return 0;
  const int ps = effective_partition(partition_size);
  const int64_t parts = std::max<int64_t>(1, ((int64_t)max_seq_len + ps - 1) / ps);
  if (parts > kMaxPartitions) return 0;
  return decode_workspace_layout(num_seqs, num_q_heads, head_dim, parts).total;
}

pa_status pa_set_decode_kernel(int32_t kernel) {
  if (kernel != PA_DECODE_KERNEL_AUTO && kernel != PA_DECODE_KERNEL_CUDA_CORES) return PA_ERR_INVALID_ARG;
  g_decode_kernel.store(kernel, std::memory_order_relaxed);
  return PA_OK;
}

}  // extern "C"

namespace pa {
namespace {
// The new tokens of a fused decode step (pa_decode_write).
struct NewTokens {
  const void *k, *v;
  int64_t stride;
  const int64_t *slots;
};

// The prefill part of a one-launch mixed step (pa_mixed_step): the prefill
// kernel's parameters as pa_prefill_chunk would pass them.
struct MixedPrefill {
  PrefillTcParams t;
  int num_chunks;
};

pa_status decode_impl(const void *q, pa_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                      const void *k_cache, const void *v_cache, const pa_kv_cache *cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
                      int32_t max_seq_len, float scale, int32_t partition_size, void *workspace,
                      size_t workspace_bytes, void *out, pa_dtype out_dtype, pa_stream_t stream,
                      const NewTokens *nt, const MixedPrefill *mix = nullptr) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  const pa_kv_cache &c = *cache;
  if (num_seqs < 0 || num_q_heads <= 0 || num_q_heads % c.num_kv_heads || max_seq_len < 0 ||
      max_blocks_per_seq <= 0 || partition_size < 0 || partition_size % 32 || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if ((st = check_q_dtype(q_dtype, c)) != PA_OK) return st;
  if (out_dtype != q_dtype && out_dtype != PA_F32) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!q || !out || !block_tables || !seq_lens || !aligned(q, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PA_ERR_INVALID_ARG;
  if ((st = check_pools(k_cache, v_cache)) != PA_OK) return st;
  if (num_seqs > kMaxDecodeRows) return PA_ERR_UNSUPPORTED;

  const int ps = effective_partition(partition_size);
  const int64_t parts64 = std::max<int64_t>(1, ((int64_t)max_seq_len + ps - 1) / ps);
  if (parts64 > kMaxPartitions) return PA_ERR_UNSUPPORTED;
  const int parts = (int)parts64;
  const int gqa = num_q_heads / c.num_kv_heads;
  const bool use_tc = g_decode_kernel.load(std::memory_order_relaxed) == PA_DECODE_KERNEL_AUTO &&
                      decode_tc_supported(c.head_dim, gqa, c.kv_dtype);
  const int hpc = use_tc ? gqa : heads_per_cta(gqa);   // query heads per work unit
  if ((double)num_seqs * parts * num_q_heads / hpc >= 2147483647.0) return PA_ERR_UNSUPPORTED;
  const WorkspaceLayout w = decode_workspace_layout(num_seqs, num_q_heads, c.head_dim, parts);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < w.total) return PA_ERR_INVALID_ARG;

  DecodeParams p{};
  p.q = q;
  p.out = out;
  p.out_f32 = out_dtype == PA_F32;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.groups = gqa / hpc;
  p.block_size = c.block_size;
  p.num_blocks = c.num_blocks;
  p.partition_size = ps;
  p.max_partitions = parts;
  const bool fp8 = c.kv_dtype == PA_FP8_E4M3;
  p.q_mult = scale * 1.4426950408889634f * (fp8 && !c.k_head_scales ? c.k_scale : 1.f);
  p.out_mult = fp8 && !c.v_head_scales ? c.v_scale : 1.f;
  p.k_hs = c.k_head_scales;
  p.v_hs = c.v_head_scales;
  char *ws = static_cast<char *>(workspace);
  p.hdr = reinterpret_cast<DecodeHeader *>(ws + w.hdr_off);
  p.items = reinterpret_cast<int32_t *>(ws + w.items_off);
  p.ws_acc = reinterpret_cast<float *>(ws + w.acc_off);
  p.ws_ml = reinterpret_cast<float2 *>(ws + w.ml_off);
  p.ws_count = reinterpret_cast<int32_t *>(ws + w.cnt_off);
  p.tile_shift = c.block_size == 32 ? 1 : 0;
  p.kv_rows = c.num_kv_heads * c.block_size;
  p.err = device_error_word();
  if (!p.err) return PA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (use_tc) {
    DecodeTcParams tp{};
    tp.d = p;
    tp.k_cache = k_cache;
    tp.v_cache = v_cache;
    tp.s_mult = p.q_mult;
    tp.k_scale = c.k_scale;
    tp.v_scale = c.v_scale;
    tp.jobs = reinterpret_cast<DecodeMergeJob *>(ws + w.jobs_off);
    if (nt) {
      tp.k_new = nt->k;
      tp.v_new = nt->v;
      tp.new_stride = nt->stride;
      tp.new_slots = nt->slots;
    }
    PoolMaps maps{};
    const bool fp8_cache = c.kv_dtype == PA_FP8_E4M3;
    if (fp8_cache ? (!encode_pool_map_fp8_blocks(&maps.k, k_cache, c) || !encode_pool_map_fp8_blocks(&maps.v, v_cache, c))
                  : (!encode_pool_map_atoms(&maps.k, k_cache, c) || !encode_pool_map_atoms(&maps.v, v_cache, c)))
      return PA_ERR_CUDA;
    if (mix) {   // the prefill tiles join the decode's grid (pa_mixed_tc.cuh)
      PrefillTcParams pt = mix->t;
      pt.err = p.err;
      if (c.kv_dtype == PA_BF16) e = launch_mixed_tc_bf16(tp, maps, pt, mix->num_chunks, gqa, s);
      else if (c.kv_dtype == PA_F16) e = launch_mixed_tc_f16(tp, maps, pt, mix->num_chunks, gqa, s);
      else if (q_dtype == PA_BF16) e = launch_mixed_tc_fp8_bf16q(tp, maps, pt, mix->num_chunks, gqa, s);
      else e = launch_mixed_tc_fp8_f16q(tp, maps, pt, mix->num_chunks, gqa, s);
      return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    if (c.kv_dtype == PA_BF16) e = launch_decode_tc_bf16(tp, gqa, c.head_dim, maps, s);
    else if (c.kv_dtype == PA_F16) e = launch_decode_tc_f16(tp, gqa, c.head_dim, maps, s);
    else if (q_dtype == PA_BF16) e = launch_decode_tc_fp8_bf16q(tp, gqa, c.head_dim, maps, s);
    else e = launch_decode_tc_fp8_f16q(tp, gqa, c.head_dim, maps, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  if (mix) return PA_ERR_INVALID_ARG;   // the caller asks for one launch only where both parts use tensor cores
  if (nt &&   // CUDA-core decode: the cache write is its own launch, just before
      launch_reshape_and_cache(nt->k, nt->v, q_dtype, num_seqs, nt->stride, nt->slots, const_cast<void *>(k_cache),
                               const_cast<void *>(v_cache), c, p.err, s) != cudaSuccess)
    return PA_ERR_CUDA;
  PoolMaps maps;
  if (!encode_pool_map(&maps.k, k_cache, c, true) || !encode_pool_map(&maps.v, v_cache, c, true))
    return PA_ERR_CUDA;
  if (c.kv_dtype == PA_BF16) e = launch_decode_bf16(p, hpc, maps, c.head_dim, s);
  else if (c.kv_dtype == PA_F16) e = launch_decode_f16(p, hpc, maps, c.head_dim, s);
  else if (q_dtype == PA_BF16) e = launch_decode_fp8_bf16q(p, hpc, maps, c.head_dim, s);
  else e = launch_decode_fp8_f16q(p, hpc, maps, c.head_dim, s);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_decode(const void *q, pa_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                    const void *k_cache, const void *v_cache, const pa_kv_cache *cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *seq_lens, int32_t max_seq_len, float scale,
                    int32_t partition_size, void *workspace, size_t workspace_bytes, void *out,
                    pa_dtype out_dtype, pa_stream_t stream) {
  return decode_impl(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, scale, partition_size, workspace, workspace_bytes, out, out_dtype, stream,
                     nullptr);
}

pa_status pa_decode_write(const void *q, pa_dtype q_dtype, int32_t num_seqs, int32_t num_q_heads,
                          const void *k_new, const void *v_new, int64_t token_stride, const int64_t *slot_mapping,
                          void *k_cache, void *v_cache, const pa_kv_cache *cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len, float scale,
                          int32_t partition_size, void *workspace, size_t workspace_bytes, void *out,
                          pa_dtype out_dtype, pa_stream_t stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (num_seqs > 0) {
    if (token_stride < (int64_t)cache->num_kv_heads * cache->head_dim || token_stride % 8) return PA_ERR_INVALID_ARG;
    if (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))
      return PA_ERR_INVALID_ARG;
  }
  const NewTokens nt{k_new, v_new, token_stride, slot_mapping};
  return decode_impl(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                     seq_lens, max_seq_len, scale, partition_size, workspace, workspace_bytes, out, out_dtype, stream,
                     &nt);
}

}  // extern "C"

namespace pa {
namespace {
// pa_prefill_chunk's argument checks.  PA_OK with *empty set: nothing to do;
// otherwise *tc tells whether the tensor-core kernel applies, and then t holds
// its parameters.
pa_status prefill_prepare(const void *q_chunk, pa_dtype q_dtype, const int32_t *cu_q_lens, const int32_t *q_start,
                          int32_t num_chunks, int32_t max_q_len, int32_t num_q_heads, const void *k_cache,
                          const void *v_cache, const pa_kv_cache *cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t max_seq_len, float scale,
                          void *out, pa_dtype out_dtype, bool *empty, bool *tc, PrefillTcParams *tp) {
  *empty = false;
  *tc = false;
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  const pa_kv_cache &c = *cache;
  if (num_chunks < 0 || max_q_len < 0 || num_q_heads <= 0 || num_q_heads % c.num_kv_heads ||
      max_seq_len < 0 || max_blocks_per_seq <= 0 || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if ((st = check_q_dtype(q_dtype, c)) != PA_OK) return st;
  if (out_dtype != q_dtype && out_dtype != PA_F32) return PA_ERR_UNSUPPORTED;
  if (num_chunks == 0 || max_q_len == 0) {
    *empty = true;
    return PA_OK;
  }
  if (!q_chunk || !out || !cu_q_lens || !q_start || !block_tables || !seq_lens ||
      !aligned(q_chunk, 16) || !aligned(out, 16) || !aligned(cu_q_lens, 4) ||
      !aligned(q_start, 4) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PA_ERR_INVALID_ARG;
  if ((st = check_pools(k_cache, v_cache)) != PA_OK) return st;
  const int64_t rows = (int64_t)num_chunks * max_q_len;
  if (rows > 2147483647ll || num_q_heads > 65535) return PA_ERR_UNSUPPORTED;
  const bool fp8 = c.kv_dtype == PA_FP8_E4M3;
  const int gqa = num_q_heads / c.num_kv_heads;
  if (prefill_tc_supported(c.head_dim, gqa)) {
    // tensor-core tiles: 128 GQA-packed rows x 128-key tiles (pa_prefill_tc.cuh)
    *tc = true;
    PrefillTcParams &t = *tp;
    t = PrefillTcParams{};
    t.q = q_chunk;
    t.k_cache = k_cache;
    t.v_cache = v_cache;
    t.out = out;
    t.out_f32 = out_dtype == PA_F32;
    t.cu_q_lens = cu_q_lens;
    t.q_start = q_start;
    t.seq_lens = seq_lens;
    t.block_tables = block_tables;
    t.max_blocks_per_seq = max_blocks_per_seq;
    t.max_q_len = max_q_len;
    t.num_q_heads = num_q_heads;
    t.num_kv_heads = c.num_kv_heads;
    t.block_size = c.block_size;
    t.num_blocks = c.num_blocks;
    t.s_mult = scale * 1.4426950408889634f * (fp8 && !c.k_head_scales ? c.k_scale : 1.f);
    t.out_mult = fp8 && !c.v_head_scales ? c.v_scale : 1.f;
    t.k_hs = c.k_head_scales;
    t.v_hs = c.v_head_scales;
  }
  return PA_OK;   // t.err is set by the caller, after every check
}
}  // namespace
}  // namespace pa

extern "C" {

pa_status pa_prefill_chunk(const void *q_chunk, pa_dtype q_dtype, const int32_t *cu_q_lens,
                           const int32_t *q_start, int32_t num_chunks, int32_t max_q_len,
                           int32_t num_q_heads, const void *k_cache, const void *v_cache,
                           const pa_kv_cache *cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *seq_lens,
                           int32_t max_seq_len, float scale, void *out, pa_dtype out_dtype,
                           pa_stream_t stream) {
  bool empty = false, use_tc = false;
  PrefillTcParams t{};
  pa_status st = prefill_prepare(q_chunk, q_dtype, cu_q_lens, q_start, num_chunks, max_q_len, num_q_heads, k_cache,
                                 v_cache, cache, block_tables, max_blocks_per_seq, seq_lens, max_seq_len, scale, out,
                                 out_dtype, &empty, &use_tc, &t);
  if (st != PA_OK || empty) return st;
  const pa_kv_cache &c = *cache;
  const int64_t rows = (int64_t)num_chunks * max_q_len;
  const bool fp8 = c.kv_dtype == PA_FP8_E4M3;
  const int gqa = num_q_heads / c.num_kv_heads;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (use_tc) {
    t.err = device_error_word();
    if (!t.err) return PA_ERR_CUDA;
    // fp8: the loaders copy whole cache blocks with bulk-tensor boxes
    PoolMaps maps{};
    if (fp8 && (!encode_pool_map_fp8_blocks(&maps.k, k_cache, c) || !encode_pool_map_fp8_blocks(&maps.v, v_cache, c)))
      return PA_ERR_CUDA;
    cudaError_t e;
    if (c.kv_dtype == PA_BF16) e = launch_prefill_tc_bf16(t, maps, gqa, num_chunks, s);
    else if (c.kv_dtype == PA_F16) e = launch_prefill_tc_f16(t, maps, gqa, num_chunks, s);
    else if (q_dtype == PA_BF16) e = launch_prefill_tc_fp8_bf16q(t, maps, gqa, num_chunks, s);
    else e = launch_prefill_tc_fp8_f16q(t, maps, gqa, num_chunks, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }

  // head_dim 64 or an uneven GQA group: one CTA per query row on the CUDA cores
  AttnParams p{};
  p.q = q_chunk;
  p.out = out;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.cu_q_lens = cu_q_lens;
  p.q_start = q_start;
  p.max_q_len = max_q_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.heads_per_cta = heads_per_cta(num_q_heads / c.num_kv_heads);
  p.block_size = c.block_size;
  p.num_blocks = c.num_blocks;
  p.partition_size = std::max(32, (max_seq_len + 31) / 32 * 32);  // one partition per row
  p.max_partitions = 1;
  p.q_mult = scale * 1.4426950408889634f * (fp8 && !c.k_head_scales ? c.k_scale : 1.f);
  p.out_mult = fp8 && !c.v_head_scales ? c.v_scale : 1.f;
  p.k_hs = c.k_head_scales;
  p.v_hs = c.v_head_scales;
  p.out_f32 = out_dtype == PA_F32;
  p.err = device_error_word();
  PoolMaps maps;
  if (!p.err || !encode_pool_map(&maps.k, k_cache, c) || !encode_pool_map(&maps.v, v_cache, c))
    return PA_ERR_CUDA;
  return dispatch_attention(q_dtype, c, p, maps, (int)rows, s) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_mixed_step(const pa_decode_part *d, const pa_prefill_part *pf, pa_dtype q_dtype, int32_t num_q_heads,
                        void *k_cache, void *v_cache, const pa_kv_cache *cache, float scale, pa_dtype out_dtype,
                        pa_stream_t stream) {
  if (!d || !pf) return PA_ERR_INVALID_ARG;
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  // every argument of the prefill part, checked as pa_prefill_chunk checks them
  bool p_empty = false, p_tc = false;
  MixedPrefill mp{};
  st = prefill_prepare(pf->q_chunk, q_dtype, pf->cu_q_lens, pf->q_start, pf->num_chunks, pf->max_q_len, num_q_heads,
                       k_cache, v_cache, cache, pf->block_tables, pf->max_blocks_per_seq, pf->seq_lens,
                       pf->max_seq_len, scale, pf->out, out_dtype, &p_empty, &p_tc, &mp.t);
  if (st != PA_OK) return st;
  mp.num_chunks = pf->num_chunks;
  // the decode part's new tokens, checked as pa_decode_write checks them
  if (d->num_seqs < 0) return PA_ERR_INVALID_ARG;
  const bool has_new = d->k_new || d->v_new || d->slot_mapping;
  if (has_new && d->num_seqs > 0) {
    if (d->token_stride < (int64_t)cache->num_kv_heads * cache->head_dim || d->token_stride % 8)
      return PA_ERR_INVALID_ARG;
    if (!d->k_new || !d->v_new || !d->slot_mapping || !aligned(d->k_new, 16) || !aligned(d->v_new, 16) ||
        !aligned(d->slot_mapping, 8))
      return PA_ERR_INVALID_ARG;
  }
  const NewTokens nt{d->k_new, d->v_new, d->token_stride, d->slot_mapping};
  const int gqa = num_q_heads / cache->num_kv_heads;   // num_q_heads checked above
  const bool one_launch = !p_empty && p_tc && d->num_seqs > 0 && mixed_tc_supported(cache->head_dim, gqa) &&
                          decode_tc_supported(cache->head_dim, gqa, cache->kv_dtype) &&
                          g_decode_kernel.load(std::memory_order_relaxed) == PA_DECODE_KERNEL_AUTO;
  st = decode_impl(d->q, q_dtype, d->num_seqs, num_q_heads, k_cache, v_cache, cache, d->block_tables,
                   d->max_blocks_per_seq, d->seq_lens, d->max_seq_len, scale, d->partition_size, d->workspace,
                   d->workspace_bytes, d->out, out_dtype, stream, has_new ? &nt : nullptr, one_launch ? &mp : nullptr);
  if (st != PA_OK || one_launch || p_empty) return st;
  return pa_prefill_chunk(pf->q_chunk, q_dtype, pf->cu_q_lens, pf->q_start, pf->num_chunks, pf->max_q_len,
                          num_q_heads, k_cache, v_cache, cache, pf->block_tables, pf->max_blocks_per_seq,
                          pf->seq_lens, pf->max_seq_len, scale, pf->out, out_dtype, stream);
}

pa_status pa_selftest_wait_timeout(pa_stream_t stream) {
  int32_t *err = device_error_word();
  if (!err) return PA_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_get_device_error(pa_stream_t stream, int32_t *code) {
  if (!code) return PA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  int32_t v = 0;
  const int32_t zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess ||
      cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess)
    return PA_ERR_CUDA;
  *code = v;
  return PA_OK;
}

const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS";
  }
  return "PA_ERR_UNKNOWN";
}

}  // extern "C"
