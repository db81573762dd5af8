// pa_noalloc.cu -- pa_decode_noalloc: paged decode with library-owned scratch.
//
// For callers that cannot allocate device memory when they decode.  The
// decode workspace (work list, split-KV partials, arrival counters) lives in a
// fixed static device array instead of caller memory; everything else is the
// ordinary pa_decode path, called unchanged with that array as its workspace.
#include <cuda.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace {

// The scratch array: one per device that loads the library, held until exit.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// The array's device address per device, with the id of the context it was
// looked up in: a device reset creates a new context (new id), in which the
// array may sit elsewhere, so the address is looked up again.
struct DeviceScratch {
  unsigned long long ctx_id;
  void *ptr;
};
std::mutex g_scratch_mu;
DeviceScratch g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Id of the context current on this thread (0: none yet).
pa_status current_context_id(unsigned long long *id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return PA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
  *id = 0;
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return PA_ERR_CUDA;
  return PA_OK;
}

// Device address of the scratch array on the current device.  The array's
// name is only a host-side handle; the runtime resolves it per device (and
// per context: the look-up is repeated after a device reset).
pa_status scratch_on_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  pa_status st = current_context_id(&id);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  DeviceScratch &s = g_scratch[dev];
  if (id == 0 || s.ptr == nullptr || s.ctx_id != id) {
    void *ptr = nullptr;
    // also binds the device's primary context to this thread if none was
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return PA_ERR_CUDA;
    if ((st = current_context_id(&id)) != PA_OK) return st;
    s.ptr = ptr;
    s.ctx_id = id;
  }
  *out = s.ptr;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void *q, pa_dtype q_dtype, int32_t num_seqs,
                                       int32_t num_q_heads, const void *k_cache,
                                       const void *v_cache, const pa_kv_cache *cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *seq_lens, int32_t max_seq_len, float scale,
                                       int32_t partition_size, void *out, pa_dtype out_dtype,
                                       pa_stream_t stream) {
  if (cache == nullptr) return PA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (num_seqs > 0) {
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, cache->num_kv_heads,
                                                  cache->head_dim, max_seq_len, partition_size);
    if (need == 0)  // invalid arguments: pa_decode reports which, before touching the device
      return pa_decode(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                       max_blocks_per_seq, seq_lens, max_seq_len, scale, partition_size, nullptr, 0,
                       out, out_dtype, stream);
    if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;  // larger than the fixed scratch
    const pa_status st = scratch_on_current_device(&scratch);
    if (st != PA_OK) return st;
  }
  // Nothing in the scratch needs clearing here: pa_decode's plan step resets
  // the work list, the scheduling cursor and the arrival counters on the
  // device before the decode kernel reads them.
  return pa_decode(q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                   max_blocks_per_seq, seq_lens, max_seq_len, scale, partition_size, scratch,
                   PA_NOALLOC_SCRATCH_BYTES, out, out_dtype, stream);
}
