// pa_common.cuh -- device helpers shared by the libpa kernels (sm_103a).
//
// Inline PTX for the Blackwell async machinery the kernels use: mbarriers,
// tiled bulk-tensor (TMA) loads into shared memory, and waits that give up
// after a bounded time instead of hanging.  Also the per-device error word
// that kernels use to report out-of-range metadata without trapping.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Device-side error word (one per device, defined in pa_api.cu and passed to
// every kernel as a pointer): the first non-zero status recorded wins; read
// and cleared by pa_get_device_error.
__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
  atomicCAS(err, 0, code);
}

// Longest a kernel waits on one mbarrier phase before it reports
// PA_ERR_TIMEOUT and abandons its work (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Arrive-and-expect for a phase whose data comes only from bulk copies: no
// earlier write of this thread needs ordering, so the arrive is relaxed.
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// records PA_ERR_TIMEOUT) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(err, PA_ERR_TIMEOUT);
      return false;
    }
  }
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled bulk-tensor load global -> shared, completion counted in bytes on
// `bar`.  x is the innermost (element) coordinate and must be a multiple of
// 16 bytes' worth of elements; y is the row.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 3D variant: coordinates (x, y, z) innermost first.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Byte offset inside a tile that the tensor map wrote with a 128-byte (or
// 64-byte) swizzle: the 16-byte chunk index (bits 4..6) is XORed with the
// 128-byte row index (bits 7..9).  The tile must start 1024-byte aligned.
template <int kSwizzleBytes>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  if constexpr (kSwizzleBytes == 128) return off ^ (((off >> 7) & 7u) << 4);
  else if constexpr (kSwizzleBytes == 64) return off ^ (((off >> 7) & 3u) << 4);
  else return off;
}

// -------------------------------------------------------------- conversions
template <typename T> struct Elem;
template <> struct Elem<__half> {
  static constexpr pa_dtype code = PA_F16;
  __device__ static float to_f32(__half x) { return __half2float(x); }
  __device__ static __half from_f32(float x) { return __float2half_rn(x); }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr pa_dtype code = PA_BF16;
  __device__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Unpack one 32-bit word holding two 16-bit floats into two fp32 values.
__device__ __forceinline__ float2 unpack2(uint32_t w, __nv_bfloat16) {
  // a bf16 is the upper half of an fp32: exact by moving bits
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ float2 unpack2(uint32_t w, __half) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
// Two e4m3 codes (low 16 bits of w) -> two fp32 values, exact (via f16).
__device__ __forceinline__ float2 unpack2_e4m3(uint32_t w16) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w16 & 0xffffu),
                                            __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Packed fp32x2 fused multiply-add: d = a * b + c on both lanes of a pair.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
        "l"(*reinterpret_cast<uint64_t *>(&c)));
  return *reinterpret_cast<float2 *>(&d);
}

// *p += v at GPU scope with acquire-release semantics; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace pa
