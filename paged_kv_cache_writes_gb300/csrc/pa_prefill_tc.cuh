// pa_prefill_tc.cuh -- chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in tensor memory), head_dim 128.
//
// What it computes ("Inside vLLM v0.7 ...", section "Architectural Blueprint
// 3: Chunked Prefill"; "High-Throughput LLM Serving with vLLM &
// PagedAttention", section "5. Chunked Prefill & Latency SLA Management"):
// row r of chunk c sits at position q_start[c] + r and attends causally to
// positions 0 .. q_start[c] + r of its paged context:
//   out[row][h] = sum_p softmax_p(scale * q[row][h] . K[p][g]) V[p][g].
// Prefill is compute-bound ("High-Throughput LLM Serving ...", section "1. The
// KV Cache Bottleneck in LLM Serving"), so Q.K^T and P.V run as dense tiles on
// the tensor pipe; the softmax stays in fp32 on the CUDA cores.
//
// Tiling.  One CTA = 128 GQA-packed query rows (128/G token rows x the G query
// heads of one KV head; packed row m = token m / G, head m % G) x every key
// tile of 64 keys up to its causal limit, so each K/V byte a CTA reads feeds
// all G heads.
//
// Roles (288 threads):
//  * warps 0-3, softmax: thread m owns packed row m = tensor-memory lane m.  It
//    reads its 64 scores of a tile with tcgen05.ld, scales and masks them,
//    keeps a lazy reference maximum (its O row in tensor memory is rescaled
//    only when a tile maximum exceeds the reference by more than 2^8), and
//    writes its row of P (16-bit, 128-byte-swizzled, K-major) for the P.V MMA.
//  * warp 4, loads: TMA boxes of 16 keys (one block-table entry) x one
//    128-byte panel into a ring of kStages K and V tiles.
//  * warps 5-7, tile preparation: fp8 tiles are widened (exactly) to the
//    query's 16-bit type; V rows past the end of the sequence are zeroed so a
//    zero probability never meets a stale (possibly NaN) value in the MMA.
//  * warp 8, MMA (one thread): S_j = Q K_j^T into one of two tensor-memory
//    score buffers, then O += P_{j-1} V_{j-1} one tile behind, so the tensor
//    pipe computes a score tile while the softmax warps work on the previous.
//
// Precision.  Q, K and V are exact in the MMA (fp8 codes widen exactly to
// bf16/f16); accumulation is fp32.  P is rounded to the 16-bit type; with a
// bf16 cache P is split into hi + lo bf16 parts (two P.V MMAs) so its
// rounding stays near 2^-16 relative, and with f16 or fp8 caches the softmax
// denominator sums the rounded P, so the output remains a convex combination
// of V rows.
//
// Every mbarrier wait is bounded (PA_ERR_TIMEOUT, then the CTA abandons its
// work); before tensor memory is freed the CTA waits for its outstanding MMAs
// and TMA copies.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

struct PrefillTcParams {
  const void *q;               // [total_q][Hq][128]
  void *out;                   // [total_q][Hq][128]
  int32_t out_f32;
  const int32_t *cu_q_lens;
  const int32_t *q_start;
  const int32_t *seq_lens;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  int32_t max_q_len;
  int32_t row_blocks;          // CTAs per chunk along the query rows
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int64_t num_blocks;
  float s_mult;                // scale * log2(e) (* k_scale for fp8)
  float out_mult;              // v_scale for fp8, else 1
  int32_t *err;
};

namespace tc {

constexpr int kD = 128;         // head_dim
constexpr int kM = 128;         // packed query rows per CTA (MMA M, tensor-memory lanes)
constexpr int kN = 64;          // keys per tile
constexpr int kStages = 3;      // K/V tiles in flight
constexpr int kThreads = 288;
constexpr float kRescaleLog2 = 8.f;

constexpr int kQBytes = kM * kD * 2;        // 2 panels x [128 rows x 128 B]
constexpr int kTileBytes = kN * kD * 2;     // 2 panels x [64 rows x 128 B]
constexpr int kTilePanel = kN * 128;        // 8 KB
constexpr int kPPanel = kM * kN * 2;        // [128 rows x 128 B] = 16 KB
constexpr int kRawBytes = kN * kD;          // fp8 tile: [64 rows x 128 B]
constexpr int kNumBars = 8 * kStages + 10;

// Shared-memory map, bytes from a 1024-aligned base (128-byte swizzle atoms).
template <bool kFp8, bool kSplit>
struct Layout {
  static constexpr int kPBuf = (kSplit ? 2 : 1) * kPPanel;  // one P buffer (hi [+ lo] panel)
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffRawK = kOffP + 2 * kPBuf;
  static constexpr int kOffRawV = kOffRawK + (kFp8 ? kStages * kRawBytes : 0);
  static constexpr int kOffBar = kOffRawV + (kFp8 ? kStages * kRawBytes : 0);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// UMMA shared-memory descriptor: 128-byte swizzle, SBO = 1024 (8 rows x 128 B).
// lbo: ignored for swizzled K-major operands (16); for an MN-major operand the
// byte distance between its 64-element panels.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (1 = bf16, 0 = f16), A K-major, B K-major or MN-major, M = 128.
__device__ __forceinline__ uint32_t umma_idesc(uint32_t ab_fmt, uint32_t n, bool b_mn_major) {
  return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((n >> 3) << 17) |
         ((uint32_t)(kM >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
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

// Bounded wait that also gives up once another role of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int32_t *err,
                                              volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// Widen 16 e4m3 codes (swizzled 16-byte chunk `ch` of raw row r) into 16
// elements of row r of the 16-bit tile (two 16-byte chunks of panel ch / 4).
template <typename QT>
__device__ __forceinline__ void widen_chunk(const uint8_t *raw_row, uint8_t *tile, int r, int ch, bool zero) {
  uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (!zero) {
    const uint4 w = *reinterpret_cast<const uint4 *>(raw_row + ((ch ^ (r & 7)) << 4));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = unpack2_e4m3(ws[i]), hi = unpack2_e4m3(ws[i] >> 16);
      o[2 * i] = pack2(lo.x, lo.y, QT{});
      o[2 * i + 1] = pack2(hi.x, hi.y, QT{});
    }
  }
  const int c0 = (2 * ch) & 7;
  uint8_t *row = tile + (ch >> 2) * kTilePanel + r * 128;
  *reinterpret_cast<uint4 *>(row + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace tc

template <typename KV, typename QT, int G>
__global__ void __launch_bounds__(tc::kThreads, 1)
    prefill_tc_kernel(const PrefillTcParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using namespace tc;
  constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  constexpr bool kBf16 = std::is_same<QT, __nv_bfloat16>::value;
  constexpr bool kSplit = kBf16 && !kFp8;   // bf16 cache: P as hi + lo
  using L = Layout<kFp8, kSplit>;
  constexpr int BR = kM / G;                // token rows per CTA
  constexpr uint32_t kAB = kBf16 ? 1u : 0u;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *k_tma = bars;                      // [kStages] TMA bytes of a K tile landed
  uint64_t *v_tma = k_tma + kStages;           // [kStages]
  uint64_t *k_ready = v_tma + kStages;         // [kStages] fp8: widened K tile written (96)
  uint64_t *v_ready = k_ready + kStages;       // [kStages] V tile ready for the MMA (96)
  uint64_t *k_free = v_ready + kStages;        // [kStages] MMA finished reading the K tile
  uint64_t *v_free = k_free + kStages;         // [kStages] MMA finished reading the V tile
  uint64_t *raw_k_free = v_free + kStages;     // [kStages] fp8: raw K tile consumed (96)
  uint64_t *raw_v_free = raw_k_free + kStages; // [kStages]
  uint64_t *s_full = raw_v_free + kStages;     // [2] score tile in tensor memory
  uint64_t *s_free = s_full + 2;               // [2] score tile read by the softmax warps (128)
  uint64_t *p_full = s_free + 2;               // [2] P tile written (128)
  uint64_t *o_done = p_full + 2;               // [2] P.V group i done -> o_done[i & 1]
  uint64_t *q_ready = o_done + 2;              // Q staged (128)
  uint64_t *fin = q_ready + 1;                 // every MMA of the CTA complete
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x / p.row_blocks, rb = blockIdx.x % p.row_blocks;
  const int g = blockIdx.y;
  const int cu0 = __ldg(p.cu_q_lens + c), nrows = __ldg(p.cu_q_lens + c + 1) - cu0;
  const int qs = __ldg(p.q_start + c);
  if (tid == 0 && g == 0 && rb == 0) {
    const int64_t len = (int64_t)qs + nrows;
    if (nrows < 0 || nrows > p.max_q_len || qs < 0 || __ldg(p.seq_lens + c) != len ||
        len > (int64_t)p.max_blocks_per_seq * p.block_size)
      record_error(p.err, PA_ERR_DEVICE_CHECK);
  }
  const int r0 = rb * BR;
  if (r0 >= nrows) return;  // whole CTA, before any barrier or tensor memory
  // keys this chunk may read: its sequence, clamped to the block table
  const int64_t cap = (int64_t)p.max_blocks_per_seq * p.block_size;
  const int64_t len64 = (int64_t)qs + nrows;
  const int seq_eff = len64 <= 0 ? 0 : (int)(len64 < cap ? len64 : cap);
  const int r_last = min(r0 + BR, nrows) - 1;
  const int kv_end = min(seq_eff, max(0, qs + r_last + 1));   // keys this CTA needs
  const int nkt = (kv_end + kN - 1) / kN;                      // key tiles (may be 0)
  const int32_t *table = p.block_tables + (int64_t)c * p.max_blocks_per_seq;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_tma[s], 1);
      mbar_init(&v_tma[s], 1);
      mbar_init(&k_ready[s], 96);
      mbar_init(&v_ready[s], 96);
      mbar_init(&k_free[s], 1);
      mbar_init(&v_free[s], 1);
      mbar_init(&raw_k_free[s], 96);
      mbar_init(&raw_v_free[s], 96);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
      mbar_init(&p_full[b], 128);
      mbar_init(&o_done[b], 1);
    }
    mbar_init(q_ready, 128);
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {  // tensor memory: S0 cols [0,64), S1 [64,128), O [128,256)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensor_map(&tmap_k);
    prefetch_tensor_map(&tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 2 * kN;

  if (warp < 4) {
    // ===================================================== softmax warps
    const int m = tid;                         // packed row = tensor-memory lane
    const int rl = m / G, hq = m % G;
    const bool row_ok = r0 + rl < nrows;
    const int head = g * G + hq;
    // keys this row attends to: positions < lim
    const int lim = row_ok ? min(seq_eff, max(0, qs + r0 + rl + 1)) : 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    {  // stage row m of Q (16-bit, 128-byte-swizzled K-major, 2 panels)
      const QT *src = static_cast<const QT *>(p.q) + ((int64_t)(cu0 + r0 + rl) * p.num_q_heads + head) * kD;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 v = row_ok ? __ldg(reinterpret_cast<const uint4 *>(src) + ch) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(smem + L::kOffQ + (ch >> 3) * (kM * 128) + m * 128 +
                                   (((ch & 7) ^ (m & 7)) << 4)) = v;
      }
    }
    fence_async_smem();
    mbar_arrive(q_ready);

    float m_ref = kNegInf, l = 0.f;
    int o_seen = 0;  // P.V groups this thread has seen complete
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait_or_abort(&s_full[b], (j >> 1) & 1, p.err, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float s[kN];
      {
        float t0[32], t1[32];
        tmem_ld32(tmem + lane_base + b * kN, t0);
        tmem_ld32(tmem + lane_base + b * kN + 32, t1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = t0[i];
          s[32 + i] = t1[i];
        }
      }
      tc_fence_before();
      mbar_arrive(&s_free[b]);
      // scale into log2 units; mask keys at or past this row's limit
      const int nvis = lim - j * kN;
      float mx[8];
#pragma unroll
      for (int i = 0; i < kN; ++i) {
        s[i] = i < nvis ? s[i] * p.s_mult : kNegInf;
        if (i < 8) mx[i] = s[i];
        else mx[i & 7] = fmaxf(mx[i & 7], s[i]);
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const bool rescale = mt > m_ref + tc::kRescaleLog2;
      const bool warp_rescale = __any_sync(0xffffffffu, rescale);
      // P buffer b was last read by P.V group j-2; rescaling O needs group j-1 done
      const int need = warp_rescale ? j - 1 : j - 2;
      while (o_seen <= need) {
        ok = __all_sync(0xffffffffu,
                        wait_or_abort(&o_done[o_seen & 1], (o_seen >> 1) & 1, p.err, abort_flag));
        if (!ok) break;
        ++o_seen;
      }
      if (!ok) break;
      if (warp_rescale) {
        const float alpha = rescale ? fast_exp2(m_ref - mt) : 1.f;
        if (j > 0) {  // O holds groups 0 .. j-1 (no group has run before tile 0)
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < kD; c0 += 32) {
            float o[32];
            tmem_ld32(tmem_o + lane_base + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem_o + lane_base + c0, o);
          }
        }
        if (rescale) {
          l *= alpha;
          m_ref = mt;
        }
      }
      // a row with nothing visible yet keeps m_ref = -inf and all s = -inf
      const float msub = m_ref == kNegInf ? 0.f : m_ref;
      uint8_t *prow = smem + L::kOffP + b * L::kPBuf + m * 128;
      float lp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pv[i] = fast_exp2(s[ch * 8 + i] - msub);  // masked: 2^-inf = 0
        uint32_t w[4], wl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[i] = pack2(pv[2 * i], pv[2 * i + 1], QT{});
          const float2 hi = unpack2(w[i], QT{});
          if constexpr (kSplit) {
            wl[i] = pack2(pv[2 * i] - hi.x, pv[2 * i + 1] - hi.y, QT{});
            lp[i] += pv[2 * i] + pv[2 * i + 1];
          } else {
            lp[i] += hi.x + hi.y;   // the rounded P that the MMA will use
          }
        }
        *reinterpret_cast<uint4 *>(prow + ((ch ^ (m & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        if constexpr (kSplit)
          *reinterpret_cast<uint4 *>(prow + kPPanel + ((ch ^ (m & 7)) << 4)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
      l += (lp[0] + lp[1]) + (lp[2] + lp[3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    // O is complete once every P.V group has finished
    while (ok && o_seen < nkt) {
      ok = __all_sync(0xffffffffu, wait_or_abort(&o_done[o_seen & 1], (o_seen >> 1) & 1, p.err, abort_flag));
      ++o_seen;
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? p.out_mult / l : 0.f;
      const int64_t obase = ((int64_t)(cu0 + r0 + rl) * p.num_q_heads + head) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        float o[32];
        if (nkt > 0) {
          tmem_ld32(tmem_o + lane_base + c0, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (!row_ok) continue;
        if (p.out_f32) {
          float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + obase + c0);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<QT *>(p.out) + obase + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(pack2(o[8 * i] * inv, o[8 * i + 1] * inv, QT{}),
                                pack2(o[8 * i + 2] * inv, o[8 * i + 3] * inv, QT{}),
                                pack2(o[8 * i + 4] * inv, o[8 * i + 5] * inv, QT{}),
                                pack2(o[8 * i + 6] * inv, o[8 * i + 7] * inv, QT{}));
        }
      }
    }
  } else if (warp == 4) {
    // ===================================================== TMA loads (lane 0 issues)
    constexpr int kSub = kN / 16;                          // 16-key boxes per tile
    constexpr int kPanels = kFp8 ? 1 : 2;
    constexpr uint32_t kBox = 16 * 128;                    // bytes per box
    int k_issued = 0, v_issued = 0;                        // tiles whose copies were issued
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int s = j % kStages;
      const uint32_t ph_prev = ((j / kStages) - 1) & 1;
      // lanes 0 .. kSub-1: block id of box `lane` (16 keys inside one block)
      const int key = j * kN + lane * 16;
      const bool has = lane < kSub && key < seq_eff;
      const int32_t blk = has ? __ldg(table + key / p.block_size) : 0;
      const bool bad = has && (blk < 0 || blk >= p.num_blocks);
      const uint32_t load_mask = __ballot_sync(0xffffffffu, has && !bad);
      const uint32_t bad_mask = __ballot_sync(0xffffffffu, bad);
      if (lane == 0 && bad_mask != 0u) record_error(p.err, PA_ERR_DEVICE_CHECK);
      const uint32_t tx = __popc(load_mask) * kPanels * kBox;
      const int32_t y = (blk * p.num_kv_heads + g) * p.block_size + (key % p.block_size);
      for (int which = 0; which < 2; ++which) {  // 0: K, 1: V
        if (lane == 0) {
          uint64_t *freed = which == 0 ? (kFp8 ? &raw_k_free[s] : &k_free[s])
                                       : (kFp8 ? &raw_v_free[s] : &v_free[s]);
          if (j >= kStages) ok = wait_or_abort(freed, ph_prev, p.err, abort_flag);
          if (ok) mbar_arrive_expect_tx_relaxed(which == 0 ? &k_tma[s] : &v_tma[s], tx);
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        if (!ok) break;
        if (which == 0) ++k_issued;
        else ++v_issued;
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          const int32_t yi = __shfl_sync(0xffffffffu, y, i);
          if (lane == 0 && ((load_mask >> i) & 1u)) {
            const CUtensorMap *map = which == 0 ? &tmap_k : &tmap_v;
            uint64_t *bar = which == 0 ? &k_tma[s] : &v_tma[s];
            const int base = which == 0 ? (kFp8 ? L::kOffRawK : L::kOffK) : (kFp8 ? L::kOffRawV : L::kOffV);
            const int stage_bytes = kFp8 ? kRawBytes : kTileBytes;
#pragma unroll
            for (int pn = 0; pn < kPanels; ++pn)
              tma_load_2d(smem + base + s * stage_bytes + pn * kTilePanel + i * kBox, map, bar, pn * 64, yi);
          }
        }
      }
    }
    // before exit: every copy issued has landed (last phase of each stage)
    if (lane == 0) {
      for (int t = max(0, k_issued - kStages); t < k_issued; ++t) mbar_wait(&k_tma[t % kStages], (t / kStages) & 1, p.err);
      for (int t = max(0, v_issued - kStages); t < v_issued; ++t) mbar_wait(&v_tma[t % kStages], (t / kStages) & 1, p.err);
      // bf16/f16 tiles: the MMA's releases of the last tiles have arrived
      if (!kFp8 && ok) {
        for (int t = max(0, nkt - kStages); t < nkt; ++t) {
          wait_or_abort(&k_free[t % kStages], (t / kStages) & 1, p.err, abort_flag);
          wait_or_abort(&v_free[t % kStages], (t / kStages) & 1, p.err, abort_flag);
        }
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ===================================================== tile preparation (96 threads)
    const int t = tid - 160;
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int s = j % kStages;
      const uint32_t ph = (j / kStages) & 1, ph_prev = ((j / kStages) - 1) & 1;
      const int valid_rows = min(kN, seq_eff - j * kN);   // V rows at or past this become zeros
      if constexpr (kFp8) {
        ok = wait_or_abort(&k_tma[s], ph, p.err, abort_flag);
        if (ok && j >= kStages) ok = wait_or_abort(&k_free[s], ph_prev, p.err, abort_flag);
        if (!ok) break;
        for (int idx = t; idx < kN * 8; idx += 96) {     // 64 rows x 8 chunks of 16 codes
          const int r = idx >> 3, ch = idx & 7;
          widen_chunk<QT>(smem + L::kOffRawK + s * kRawBytes + r * 128, smem + L::kOffK + s * kTileBytes, r, ch,
                          false);
        }
        fence_async_smem();
        mbar_arrive(&raw_k_free[s]);
        mbar_arrive(&k_ready[s]);
        ok = wait_or_abort(&v_tma[s], ph, p.err, abort_flag);
        if (ok && j >= kStages) ok = wait_or_abort(&v_free[s], ph_prev, p.err, abort_flag);
        if (!ok) break;
        for (int idx = t; idx < kN * 8; idx += 96) {
          const int r = idx >> 3, ch = idx & 7;
          widen_chunk<QT>(smem + L::kOffRawV + s * kRawBytes + r * 128, smem + L::kOffV + s * kTileBytes, r, ch,
                          r >= valid_rows);
        }
        fence_async_smem();
        mbar_arrive(&raw_v_free[s]);
        mbar_arrive(&v_ready[s]);
      } else {
        // V landed in the MMA tile itself; zero its rows past the sequence end
        ok = wait_or_abort(&v_tma[s], ph, p.err, abort_flag);
        if (!ok) break;
        if (valid_rows < kN) {
          for (int idx = t; idx < (kN - valid_rows) * 16; idx += 96) {
            const int r = valid_rows + (idx >> 4), ch = idx & 15;
            *reinterpret_cast<uint4 *>(smem + L::kOffV + s * kTileBytes + (ch >> 3) * kTilePanel + r * 128 +
                                       ((ch & 7) << 4)) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
        }
        mbar_arrive(&v_ready[s]);
      }
    }
    // fp8: the MMA's releases of the last widened tiles have arrived
    if (kFp8 && ok) {
      for (int tt = max(0, nkt - kStages); tt < nkt; ++tt) {
        wait_or_abort(&k_free[tt % kStages], (tt / kStages) & 1, p.err, abort_flag);
        wait_or_abort(&v_free[tt % kStages], (tt / kStages) & 1, p.err, abort_flag);
      }
    }
  } else {
    // ===================================================== MMA issue (warp 8, lane 0)
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc(kAB, kN, false);
      const uint32_t idesc_o = umma_idesc(kAB, kD, true);
      bool ok = nkt == 0 || wait_or_abort(q_ready, 0, p.err, abort_flag);
      auto pv = [&](int i) {  // O += P_i V_i
        const int s = i % kStages, b = i & 1;
        ok = ok && wait_or_abort(&p_full[b], (i >> 1) & 1, p.err, abort_flag);
        ok = ok && wait_or_abort(&v_ready[s], (i / kStages) & 1, p.err, abort_flag);
        if (!ok) return;
        tc_fence_after();
        const uint32_t pbase = smem_u32(smem + L::kOffP + b * L::kPBuf);
        const uint32_t vbase = smem_u32(smem + L::kOffV + s * kTileBytes);
#pragma unroll
        for (int half = 0; half < (kSplit ? 2 : 1); ++half) {
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            const uint64_t ad = umma_desc(pbase + half * kPPanel + kk * 32, 16);
            const uint64_t bd = umma_desc(vbase + kk * 16 * 128, kTilePanel);
            umma(tmem_o, ad, bd, idesc_o, (i > 0 || half > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&o_done[b]);
        umma_commit(&v_free[s]);
      };
      if (ok) tc_fence_after();
      const uint32_t qbase = smem_u32(smem + L::kOffQ);
      for (int j = 0; j < nkt && ok; ++j) {
        const int s = j % kStages, b = j & 1;
        ok = kFp8 ? wait_or_abort(&k_ready[s], (j / kStages) & 1, p.err, abort_flag)
                  : wait_or_abort(&k_tma[s], (j / kStages) & 1, p.err, abort_flag);
        if (ok && j >= 2) ok = wait_or_abort(&s_free[b], ((j - 2) >> 1) & 1, p.err, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kbase = smem_u32(smem + L::kOffK + s * kTileBytes);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint64_t ad = umma_desc(qbase + (k >> 2) * (kM * 128) + (k & 3) * 32, 16);
          const uint64_t bd = umma_desc(kbase + (k >> 2) * kTilePanel + (k & 3) * 32, 16);
          umma(tmem + b * kN, ad, bd, idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        umma_commit(&k_free[s]);
        if (j >= 1) pv(j - 1);
      }
      if (ok && nkt > 0) pv(nkt - 1);
      // every MMA issued above is complete before tensor memory is freed
      umma_commit(fin);
      mbar_wait(fin, 0, p.err);
    }
    __syncwarp();
  }

  // ===================================================== teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tmem));
  }
}

// Host launcher: grid (chunks x row blocks, KV heads), 288 threads, one CTA per SM.
template <typename KV, typename QT, int G>
cudaError_t launch_prefill_tc_one(const PrefillTcParams &p0, const PoolMaps &m, int num_chunks, cudaStream_t s) {
  constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  constexpr bool kSplit = std::is_same<QT, __nv_bfloat16>::value && !kFp8;
  constexpr int smem = tc::Layout<kFp8, kSplit>::kSmemBytes;
  PrefillTcParams p = p0;
  p.row_blocks = (p.max_q_len + (tc::kM / G) - 1) / (tc::kM / G);
  auto kern = prefill_tc_kernel<KV, QT, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t gx = (int64_t)num_chunks * p.row_blocks;
  if (gx > 2147483647ll || p.num_kv_heads > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)gx, (unsigned)p.num_kv_heads);
  kern<<<grid, tc::kThreads, smem, s>>>(p, m.k, m.v);
  return cudaGetLastError();
}

template <typename KV, typename QT>
cudaError_t launch_prefill_tc(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks, cudaStream_t s) {
  switch (gqa) {
    case 1: return launch_prefill_tc_one<KV, QT, 1>(p, m, num_chunks, s);
    case 2: return launch_prefill_tc_one<KV, QT, 2>(p, m, num_chunks, s);
    case 4: return launch_prefill_tc_one<KV, QT, 4>(p, m, num_chunks, s);
    case 8: return launch_prefill_tc_one<KV, QT, 8>(p, m, num_chunks, s);
    case 16: return launch_prefill_tc_one<KV, QT, 16>(p, m, num_chunks, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
