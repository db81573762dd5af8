// pa_tcgen05.cuh -- inline-PTX helpers for the 5th-generation tensor cores
// (sm_103a) shared by the tensor-core attention kernels: UMMA shared-memory
// and instruction descriptors, tcgen05.mma / commit / ld / st, the fences
// between the generic and async proxies, elected-lane issue, bounded waits
// that honour a CTA-wide abort flag, 16-byte cp.async with zero-fill, the
// exact e4m3 -> 16-bit widening used to feed fp8 caches to kind::f16, and
// the two-term e4m3 split of fp32 operands for kind::f8f6f4.
#pragma once

#include <type_traits>

#include "pa_common.cuh"

namespace pa {
namespace tc {

// UMMA shared-memory descriptor: 128-byte swizzle, SBO = 1024 (8 rows x 128 B).
// lbo: ignored for swizzled K-major operands (16); for an MN-major operand the
// byte distance between its 64-element panels.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// The same with the stride between 8-row groups (SBO) given, for operands
// whose 1024-byte swizzle atoms are not packed back to back.
__device__ __forceinline__ uint64_t umma_desc_sbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// UMMA shared-memory descriptor with the 64-byte swizzle (8 rows x 64 B per
// 512-byte atom), for operands whose rows are 64 bytes: fp8 with head_dim 64.
__device__ __forceinline__ uint64_t umma_desc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)4 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (1 = bf16, 0 = f16), each K-major or MN-major (transposed), M = 128.
__device__ __forceinline__ uint32_t umma_idesc(uint32_t ab_fmt, uint32_t n, bool b_mn_major, bool a_mn_major = false) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The same with 8-bit operands (kind::f8f6f4; an instruction descriptor whose
// A and B formats are 0 selects e4m3 x e4m3), K = 32 per instruction.
__device__ __forceinline__ void umma_f8(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// x -> two e4m3 codes with x = hi + lo / 16 + err: hi = e4m3(x), lo =
// e4m3(16 (x - hi)) (round to nearest even; x - hi is exact in fp32).  For
// |x| <= 256, |err| <= 2^-8 |x| + 2^-14 (hi is within 2^-4 |x| of x, lo
// within 2^-4 of its argument or half of e4m3's subnormal step 2^-9), and
// nothing saturates.  Two values at a time: bytes (x0, x1) of each 16-bit result.
__device__ __forceinline__ void split2_e4m3(float2 x, uint32_t &hi, uint32_t &lo) {
  hi = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
  const float2 h = unpack2_e4m3(hi);
  lo = __nv_cvt_float2_to_fp8x2(make_float2((x.x - h.x) * 16.f, (x.y - h.y) * 16.f), __NV_SATFINITE, __NV_E4M3);
}

// x -> three e4m3 codes with x = hi + mid / 16 + lo / 256 + err: the two-term
// split of 16 (x - hi) after hi.  Every f16 value with 2^-7 <= |x| <= 256 is
// held exactly (its 11 significant bits fit in three terms), any smaller one
// to 2^-18.  (Two terms hold every bf16 value with |x| >= 2^-6 exactly.)
// Bytes (x0, x1) of each result.
__device__ __forceinline__ void split3_e4m3(float2 x, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
  hi = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
  const float2 h = unpack2_e4m3(hi);
  const float2 r = make_float2((x.x - h.x) * 16.f, (x.y - h.y) * 16.f);
  split2_e4m3(r, mid, lo);
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far is complete.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes -> visible to the async proxy (MMA operand reads).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's tensor-memory lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive 32-bit columns of this thread's tensor-memory lane (warp-collective).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// A operand in tensor memory (P): O[tmem_d] (+)= A[tmem_a] * B[desc].
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two fp32 -> packed 16-bit pair of the query type (round to nearest even).
__device__ __forceinline__ uint32_t pack2(float a, float b, __nv_bfloat16) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack2(float a, float b, __half) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// True in exactly one lane of the (fully active) warp, the same lane every time.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred != 0;
}

// bf16 bits of a non-negative-or-any finite fp32 value rounded to 8 significant
// bits (ties away from zero), kept in the upper half of the fp32 bit pattern
// so that the result is also the rounded value as an fp32.
__device__ __forceinline__ uint32_t bf16_round_bits(float x) {
  return (__float_as_uint(x) + 0x8000u) & 0xffff0000u;
}
// Pack the upper halves of two fp32 bit patterns into one bf16x2 word (a low, b high).
__device__ __forceinline__ uint32_t pack_hi_halves(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Bounded wait that also gives up once another role of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int32_t *err,
                                              volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// 16-byte global -> shared copy that bypasses L1; src_bytes 0 writes zeros
// (and reads nothing).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
// One arrival on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in the barrier's initial count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_nc16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16 e4m3 codes (one 16-byte word) -> 16 elements of the query's 16-bit type,
// exactly (e4m3 -> f16 is exact, and every e4m3 value is a bf16 value).
template <typename QT>
__device__ __forceinline__ void widen16(uint4 w, uint32_t (&o)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (std::is_same<QT, __half>::value) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(ws[i] & 0xffffu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(ws[i] >> 16), __NV_E4M3);
      o[2 * i] = *reinterpret_cast<const uint32_t *>(&lo);
      o[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&hi);
    } else {
      // every e4m3 value is a bf16 value: the upper halves of the fp32 patterns are exact
      const float2 lo = unpack2_e4m3(ws[i]), hi = unpack2_e4m3(ws[i] >> 16);
      o[2 * i] = __byte_perm(__float_as_uint(lo.x), __float_as_uint(lo.y), 0x7632);
      o[2 * i + 1] = __byte_perm(__float_as_uint(hi.x), __float_as_uint(hi.y), 0x7632);
    }
  }
}

// 4D tiled bulk-tensor load global -> shared, coordinates innermost first,
// completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

}  // namespace tc
}  // namespace pa
