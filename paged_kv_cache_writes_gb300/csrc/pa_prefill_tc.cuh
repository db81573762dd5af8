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
// Tiling.  One CTA = one or two Q tiles of 128 GQA-packed query rows (128/G
// token rows per tile x the G query heads of one KV head; packed row m =
// token m / G, head m % G; tile m / 128) x every key tile of 128 keys up to
// its causal limit.  Each K/V tile feeds every Q tile and all G heads.
//
// Roles (416 threads with two Q tiles, 288 with one):
//  * warps 0-3 / 4-7, softmax of Q tile 0 / 1: thread m owns packed row m
//    (tensor-memory lane m % 128).  It reads its 128 scores with tcgen05.ld
//    twice (maximum, then probabilities), masks them on tiles that reach its
//    causal limit, keeps a lazy reference maximum (its O row in tensor memory
//    is rescaled only when a tile maximum exceeds the reference by more than
//    2^8), and writes P (16-bit pairs) back over the scores with tcgen05.st,
//    each 16 keys' P into those keys' own 16 columns (hi pairs, then lo
//    pairs for a bf16 cache): the P.V MMA reads P straight from tensor
//    memory.
//  * the next 4 warps load: each warp gathers 32 rows (two runs of 16 keys,
//    each inside one block of the block table) of every K and V tile into a
//    ring of kStages tiles, 512 contiguous bytes per warp instruction.
//    16-bit caches: 16-byte cp.async straight into the 128-byte-swizzled MMA
//    layout; fp8 caches, one Q tile per CTA: each warp brings its rows'
//    cache blocks (one bulk-tensor box per block) into a ring of code tiles
//    two tiles ahead, then widens them exactly to f16 from shared memory
//    into the MMA layout; with two Q tiles (no shared memory to spare):
//    register loads half a tile ahead, widened on the way to shared memory.
//    Rows past the end of the sequence are
//    zero-filled so a zero probability never meets a stale (possibly NaN)
//    value in the MMA.
//  * last warp, MMA (one elected lane issues): for each Q tile t in turn,
//    O_t += P_t(j) V_j as soon as P_t(j) is written, then S_t(j+1) = Q_t
//    K_{j+1}^T into the same buffer once that P.V has completed; with two Q
//    tiles, one tile's MMAs run while the other tile's softmax works.
//
// Precision.  K and V are exact in the MMA; accumulation is fp32.  With a
// 16-bit cache the MMAs take the cache's type and Q is exact.  With an fp8
// cache they take f16 operands: the codes widen to f16 exactly (one
// conversion per pair, where bf16 would take three), and bf16 query rows are
// each multiplied by a power of two 2^e that puts the row's largest element
// in [2^14, 2^15) and rounded to f16, exact for every element above 2^-28 of
// that largest one (bf16 has 8 significant bits, f16 11); the scores are
// multiplied back by 2^-e in the softmax.  P must be 16-bit in the MMA: with
// a bf16 cache P is split into hi + lo bf16 parts (two P.V MMAs) that sum to
// P within 2^-16 relative; otherwise P is rounded once to f16 (to nearest
// even) and the softmax denominator sums the rounded P, so the output
// remains a convex combination of V rows.
//
// Every mbarrier wait is bounded (PA_ERR_TIMEOUT, then the CTA abandons its
// work); before tensor memory is freed the CTA waits for its outstanding MMAs
// and copies.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

struct PrefillTcParams {
  const void *q;               // [total_q][Hq][128]
  const void *k_cache;         // [num_blocks][Hkv][block_size][128]
  const void *v_cache;
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
  float s_mult;                // scale * log2(e) (* k_scale for fp8); a negative value flips q's sign
  float out_mult;              // v_scale for fp8, else 1
  const float *k_hs;           // fp8, optional: [Hkv] per-head scales multiplying s_mult / out_mult
  const float *v_hs;
  int32_t *err;
};

namespace tc {

// p0, p1 -> one f16x2 word (p0 in the low half), each rounded to nearest
// even by the conversion pipe; the two rounded values, widened exactly, are
// added to acc on the FMA pipe (mixed-precision fma with f16 sources).  The
// integer pipe, which the masks, maxima and addressing keep busy, is left
// alone.
__device__ __forceinline__ uint32_t f16x2_rn_add(float p0, float p1, float2 &acc) {
  uint32_t w;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(p1), "f"(p0));
  unsigned short lo, hi;
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
  const unsigned short one = 0x3c00;   // f16 1.0
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc.x) : "h"(lo), "h"(one));
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc.y) : "h"(hi), "h"(one));
  return w;
}

constexpr int kD = 128;         // head_dim
constexpr int kM = 128;         // packed query rows per Q tile (MMA M, tensor-memory lanes)
constexpr int kN = 128;         // keys per tile
constexpr int kStages = 2;      // K/V tiles in flight

// Warp roles and tensor-memory size for a CTA of QT Q tiles (1 or 2).
template <int QT>
struct Roles {
  static constexpr int kSoftmax = QT * 128;           // softmax threads (warps 0 .. 4*QT-1)
  static constexpr int kLoadWarp0 = kSoftmax / 32;    // the next 4 warps load
  static constexpr int kMmaWarp = kLoadWarp0 + 4;     // the last warp issues the MMAs
  static constexpr int kThreads = (kMmaWarp + 1) * 32;
  // score/P buffers of 128 columns per Q tile: two with one Q tile (the next
  // scores are computed while the softmax works), one with two Q tiles
  static constexpr int kBufs = QT == 1 ? 2 : 1;
  static constexpr int kTmemCols = 512;               // QT*kBufs*128 score/P columns, then QT*128 of O
};
constexpr float kRescaleLog2 = 8.f;

constexpr int kQBytes = kM * kD * 2;        // one Q tile: 2 panels x [128 rows x 128 B]
constexpr int kTileBytes = kN * kD * 2;     // 2 panels x [128 rows x 128 B]
constexpr int kTilePanel = kN * 128;        // 16 KB
constexpr int kLoaders = 128;               // threads of the load warps
constexpr int kCodeTile = kN * kD;          // fp8 codes of one K or V tile (128 rows x 128 B)
constexpr int kMaxCodeStages = 2;
constexpr int kNumBars = 4 * kStages + 3 * 4 + 2 + 4 * kMaxCodeStages;

// Shared-memory map, bytes from a 1024-aligned base (128-byte swizzle atoms).
// fp8 caches with one Q tile: kCStages tiles of codes (K then V) after the
// 16-bit K/V stages.
template <int QT, bool kFp8 = false>
struct Layout {
  static constexpr int kCStages = (kFp8 && QT == 1) ? kMaxCodeStages : 0;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + QT * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffCode = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffCode + kCStages * 2 * kCodeTile;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kOffCode % 1024 == 0 && kCodeTile % 1024 == 0, "1024-byte swizzle atoms for the code boxes");
};

}  // namespace tc

// The prefill CTA (chunk x row block bx, KV head by), for prefill_tc_kernel and
// for the prefill CTAs of the mixed kernel (pa_mixed_tc.cuh).
template <typename KV, typename QT, int G, int kQTiles>
__device__ __forceinline__ void prefill_tc_body(const PrefillTcParams &p, int bx, int by, const CUtensorMap *tmap_k,
                                                const CUtensorMap *tmap_v) {
  using namespace tc;
  using L = Layout<kQTiles, std::is_same<KV, uint8_t>::value>;
  using R = Roles<kQTiles>;
  constexpr int kSoftmax = R::kSoftmax, kLoadWarp0 = R::kLoadWarp0, kMmaWarp = R::kMmaWarp;
  constexpr int kTmemCols = R::kTmemCols;
  constexpr int kBufs = R::kBufs;
  constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  constexpr bool kBf16 = std::is_same<QT, __nv_bfloat16>::value;
  constexpr bool kSplit = kBf16 && !kFp8;   // bf16 cache: P as hi + lo
  constexpr int BR = kQTiles * kM / G;      // token rows per CTA
  constexpr bool kF16Ops = kFp8 || !kBf16;   // f16 MMA operands (f16 cache, or any fp8 cache)
  constexpr uint32_t kAB = kF16Ops ? 0u : 1u;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
  uint64_t *k_full = bars;                       // [kStages] K tile in shared memory (128 loader arrivals)
  uint64_t *v_full = k_full + kStages;           // [kStages] V tile (128)
  uint64_t *k_free = v_full + kStages;           // [kStages] MMAs finished reading the K tile
  uint64_t *v_free = k_free + kStages;           // [kStages] MMAs finished reading the V tile
  uint64_t *s_full = v_free + kStages;           // [tile][buf] scores of key tile j in buffer j % kBufs
  uint64_t *p_full = s_full + 4;                 // [tile][buf] P of key tile j written over them (128 arrivals)
  uint64_t *o_done = p_full + 4;                 // [tile] P.V of key tile j complete (phase j)
  uint64_t *q_ready = o_done + 4;                // Q staged (every softmax thread)
  uint64_t *fin = q_ready + 1;                   // every MMA of the CTA complete
  uint64_t *code_full = fin + 1;                 // [load warp][code stage] the warp's fp8 boxes landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = bx / p.row_blocks, rb = bx % p.row_blocks;
  const int g = by;
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
      mbar_init(&k_full[s], kLoaders);
      mbar_init(&v_full[s], kLoaders);
      mbar_init(&k_free[s], 1);
      mbar_init(&v_free[s], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(q_ready, kSoftmax);
    mbar_init(fin, 1);
    for (int i = 0; i < 4 * kMaxCodeStages; ++i) mbar_init(&code_full[i], 1);   // one expect-tx arrival
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // columns: tile t's score/P buffer b at (t*kBufs + b)*128; tile t's O after all of them
  auto sbuf = [&](int t, int b) { return tmem + (uint32_t)((t * kBufs + b) * kN); };
  auto obuf = [&](int t) { return tmem + (uint32_t)(kQTiles * kBufs * kN + t * kD); };

  if (warp < kLoadWarp0) {
    // ===================================================== softmax warps (Q tile t = warp / 4)
    const int m = tid;                         // packed row
    const int t = m / kM;
    const int rl = m / G, hq = m % G;
    const bool row_ok = r0 + rl < nrows;
    const int head = g * G + hq;
    // keys this row attends to: positions < lim
    const int lim = row_ok ? min(seq_eff, max(0, qs + r0 + rl + 1)) : 0;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // scores are scaled by |s_mult| in the exponent; a negative scale flips q's sign instead
    float cmul = fabsf(p.s_mult) * (p.k_hs ? __ldg(p.k_hs + g) : 1.f);
    const uint32_t qflip = p.s_mult < 0.f ? 0x80008000u : 0u;
    {  // stage row m of Q (16-bit, 128-byte-swizzled K-major, 2 panels per tile)
      const QT *src = static_cast<const QT *>(p.q) + ((int64_t)(cu0 + r0 + rl) * p.num_q_heads + head) * kD;
      const int mr = m % kM;
      uint8_t *qt = smem + L::kOffQ + t * kQBytes;
      if constexpr (kFp8 && kBf16) {
        // f16 operands: the row times 2^e (its largest element in [2^14, 2^15)), rounded to f16;
        // the scores are multiplied back by 2^-e
        uint4 v[16];
        float amax = 0.f;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          v[ch] = row_ok ? __ldg(reinterpret_cast<const uint4 *>(src) + ch) : make_uint4(0, 0, 0, 0);
          const uint32_t ws[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(__uint_as_float((ws[i] << 16) & 0x7fffffffu),
                                     __uint_as_float(ws[i] & 0x7fff0000u)));   // NaN ignored
        }
        const int eb = max(1, (int)((__float_as_uint(amax) >> 23) & 0xff));
        const int e = amax > 0.f ? max(-126, min(126, 141 - eb)) : 0;
        const float sc = __uint_as_float((uint32_t)(e + 127) << 23);
        cmul *= __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint32_t ws[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = unpack2(ws[i], __nv_bfloat16{});
            const __half2 h = __floats2half2_rn(f.x * sc, f.y * sc);
            o[i] = *reinterpret_cast<const uint32_t *>(&h) ^ qflip;
          }
          *reinterpret_cast<uint4 *>(qt + (ch >> 3) * (kM * 128) + mr * 128 + (((ch & 7) ^ (mr & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          uint4 v = row_ok ? __ldg(reinterpret_cast<const uint4 *>(src) + ch) : make_uint4(0, 0, 0, 0);
          v.x ^= qflip; v.y ^= qflip; v.z ^= qflip; v.w ^= qflip;
          *reinterpret_cast<uint4 *>(qt + (ch >> 3) * (kM * 128) + mr * 128 + (((ch & 7) ^ (mr & 7)) << 4)) = v;
        }
      }
    }
    fence_async_smem();
    mbar_arrive(q_ready);

    float m_ref = kNegInf;                     // reference maximum, log2 units
    float2 lacc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};   // partial row sums
    const float2 ones = make_float2(1.f, 1.f);
    bool ok = true;
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p.err, abort_flag));
    };
    for (int j = 0; j < nkt; ++j) {
      const int b = j % kBufs;
      ok = wait_all(&s_full[t * kBufs + b], (j / kBufs) & 1);
      if (!ok) break;
      const uint32_t sb = sbuf(t, b) + lane_base;
      tc_fence_after();
      // keys at or past this row's limit are masked, but only tiles that reach
      // some row's limit (the causal diagonal, the sequence end) need the test
      const int nvis = lim - j * kN;
      const bool full_tile = __all_sync(0xffffffffu, nvis >= kN);
      // pass 1: the tile maximum
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = kNegInf;
#pragma unroll
      for (int ck = 0; ck < kN / 32; ++ck) {
        float sv[32];
        tmem_ld32(sb + 32 * ck, sv);
        if (!full_tile) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * ck + i >= nvis) sv[i] = kNegInf;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) mx[i & 7] = fmax3(mx[i & 7], sv[2 * i], sv[2 * i + 1]);
      }
      const float mr = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mt = mr == kNegInf ? kNegInf : mr * cmul;   // tile maximum, log2 units
      const bool rescale = mt > m_ref + tc::kRescaleLog2;
      if (__any_sync(0xffffffffu, rescale)) {
        const float alpha = rescale ? fast_exp2(m_ref - mt) : 1.f;
        if (j > 0) {
          // O holds the P.V of tiles 0 .. j-1: wait for the last of them, then rescale in place
          ok = wait_all(&o_done[t], (j - 1) & 1);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < kD; c0 += 32) {
            float o[32];
            tmem_ld32(obuf(t) + lane_base + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(obuf(t) + lane_base + c0, o);
          }
        }
        if (rescale) {
#pragma unroll
          for (int i = 0; i < 4; ++i) lacc[i] = make_float2(lacc[i].x * alpha, lacc[i].y * alpha);
          m_ref = mt;
        }
      }
      // pass 2: p = 2^(s * |s_mult| - m_ref), 16 keys at a time, written over
      // those keys' own 16 score columns.  A row with nothing visible yet keeps
      // m_ref = -inf.
      const float msub = m_ref == kNegInf ? 0.f : m_ref;
      const float2 cc = make_float2(cmul, cmul), nm = make_float2(-msub, -msub);
#pragma unroll 1
      for (int ck = 0; ck < kN / 32; ++ck) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {   // keys 32ck + 16hh .. +15
          float sv[16];
          tmem_ld16(sb + 32 * ck + 16 * hh, sv);
          uint32_t w[8], wl[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int i0 = 32 * ck + 16 * hh + 2 * k;
            const float2 a = ffma2(make_float2(sv[2 * k], sv[2 * k + 1]), cc, nm);
            float2 pk = make_float2(fast_exp2(a.x), fast_exp2(a.y));
            if (!full_tile) {
              if (i0 >= nvis) pk.x = 0.f;
              if (i0 + 1 >= nvis) pk.y = 0.f;
            }
            if constexpr (kSplit) {
              // bf16 cache: hi = p rounded to bf16, lo = p - hi (exact in fp32) rounded to
              // bf16, both by the conversion pipe; hi + lo is within 2^-16 of p, and the
              // denominator sums p itself
              uint32_t hw, lw2;
              asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hw) : "f"(pk.y), "f"(pk.x));
              w[k] = hw;
              const float2 lo = ffma2(make_float2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xffff0000u)),
                                      make_float2(-1.f, -1.f), pk);
              asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lw2) : "f"(lo.y), "f"(lo.x));
              wl[k] = lw2;
              lacc[k & 3] = ffma2(pk, ones, lacc[k & 3]);
            } else {
              // f16 P (p <= 2^8), rounded to nearest even; the denominator sums the rounded P
              w[k] = f16x2_rn_add(pk.x, pk.y, lacc[k & 3]);
            }
          }
          // P of these 16 keys goes over their own 16 score columns (read just
          // above): hi words in the first 8, lo words (bf16 cache) in the next 8
          tmem_st8(sb + 32 * ck + 16 * hh, w);
          if constexpr (kSplit) tmem_st8(sb + 32 * ck + 16 * hh + 8, wl);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[t * kBufs + b]);
    }
    const float l = ((lacc[0].x + lacc[0].y) + (lacc[1].x + lacc[1].y)) +
                    ((lacc[2].x + lacc[2].y) + (lacc[3].x + lacc[3].y));
    // O is complete once the tile's last P.V has finished
    if (ok && nkt > 0) ok = wait_all(&o_done[t], (nkt - 1) & 1);
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? p.out_mult * (p.v_hs ? __ldg(p.v_hs + g) : 1.f) / l : 0.f;
      const int64_t obase = ((int64_t)(cu0 + r0 + rl) * p.num_q_heads + head) * kD;
#pragma unroll 1
      for (int c0 = 0; c0 < kD; c0 += 32) {
        float o[32];
        if (nkt > 0) {
          tmem_ld32(obuf(t) + lane_base + c0, o);
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
  } else if (warp < kMmaWarp) {
    // ===================================================== loaders (4 warps)
    // Warp lw fills rows 32*lw .. 32*lw+31 of every K and V tile: two runs of
    // 16 keys, each inside one block of the block table (tiles start at
    // multiples of 128, blocks hold 16 or 32 keys).
    const int lw = warp - kLoadWarp0;
    constexpr int kRowBytes = kFp8 ? kD : 2 * kD;
    const char *kpool = static_cast<const char *>(p.k_cache);
    const char *vpool = static_cast<const char *>(p.v_cache);
    int32_t win = -1;                 // lane l: block id of run (l & 1) of tile win_base + (l >> 1)
    int win_base = -16;
    // block id of this warp's run r (0/1) of tile j (warp-uniform); -1 past the sequence
    auto block_of = [&](int j, int r) -> int32_t {
      if (j - win_base >= 16) {
        win_base = j;
        const int jt = j + (lane >> 1);
        const int key = jt * kN + 32 * lw + 16 * (lane & 1);
        win = -1;
        if (jt < nkt && key < seq_eff) {
          const int32_t bi = __ldg(table + key / p.block_size);
          if (bi < 0 || bi >= p.num_blocks) record_error(p.err, PA_ERR_DEVICE_CHECK);
          else win = bi;
        }
      }
      return __shfl_sync(0xffffffffu, win, 2 * (j - win_base) + r);
    };
    // first cache row of run r's 16 keys in tile j, and how many of them hold data
    auto rows_of = [&](int j, int r, int64_t &row0) -> int {
      const int key0 = j * kN + 32 * lw + 16 * r;
      const int32_t blk = block_of(j, r);
      row0 = ((int64_t)max(blk, 0) * p.num_kv_heads + g) * p.block_size + (key0 % p.block_size);
      return blk < 0 ? 0 : min(16, seq_eff - key0);
    };
    bool ok = true;
    auto wait_slot = [&](uint64_t *bar, uint32_t parity) {
      ok = __all_sync(0xffffffffu, wait_or_abort(bar, parity, p.err, abort_flag));
      return ok;
    };
    if constexpr (!kFp8) {
      // 16-bit rows (256 B): per instruction 2 rows x 16 chunks of 16 B
      const int q = lane & 15, pn = q >> 3, cq = q & 7;
      for (int j = 0; j < nkt && ok; ++j) {
        const int s = j % kStages;
        const uint32_t ph_prev = ((j / kStages) - 1) & 1;
        int64_t row0[2];
        int nval[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) nval[r] = rows_of(j, r, row0[r]);
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          if (j >= kStages && !wait_slot(which ? &v_free[s] : &k_free[s], ph_prev)) break;
          const char *pool = which ? vpool : kpool;
          uint8_t *tile = smem + (which ? L::kOffV : L::kOffK) + s * kTileBytes + pn * kTilePanel;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = 2 * i + (lane >> 4);             // row among the run's 16
              const int row = 32 * lw + 16 * r + rr;           // row of the tile
              const bool v = rr < nval[r];
              const char *src = v ? pool + (row0[r] + rr) * kRowBytes + q * 16 : pool;
              cp_async16(tile + row * 128 + ((cq ^ (row & 7)) << 4), src, v ? 16u : 0u);
            }
          }
          cp_async_arrive_noinc(which ? &v_full[s] : &k_full[s]);
        }
      }
    } else if constexpr (L::kCStages > 0) {
      // fp8, one Q tile: warp lw's rows of tile j are one or two whole cache
      // blocks (block_size 32 or 16) of K and of V; it copies them with one
      // bulk-tensor box each into code stage j % kCS (128-byte swizzle, as in
      // the pool map) kCS tiles ahead, then widens them to f16 into the K/V
      // stage.  Each warp waits only for its own boxes.
      constexpr int kCS = L::kCStages;
      const int q = lane & 7, pn = q >> 2, c0 = (2 * q) & 7;
      const int bs = p.block_size;
      uint64_t *cbar = code_full + lw * kCS;
      int issued = 0;      // tiles whose boxes this warp has issued
      uint32_t nvs = 0;    // byte 2 * stage + run: rows of that run holding keys (the block-id window only moves forward)
      auto issue_codes = [&](int j) {
        const int cs = j % kCS;
        int64_t row0;
        const uint32_t n0 = (uint32_t)rows_of(j, 0, row0), n1 = (uint32_t)rows_of(j, 1, row0);
        nvs = (nvs & ~(0xffffu << (16 * cs))) | ((n0 | (n1 << 8)) << (16 * cs));
        const int32_t b0 = block_of(j, 0), b1 = bs == 16 ? block_of(j, 1) : -1;
        const uint32_t n = (b0 >= 0 ? 1u : 0u) + (b1 >= 0 ? 1u : 0u);
        if (lane == 0) mbar_arrive_expect_tx(&cbar[cs], n * 2u * (uint32_t)(bs * kD));
        __syncwarp();
        if (lane < 4) {   // lane = 2 * which + run
          const int which = lane >> 1, r = lane & 1;
          const int32_t blk = r ? b1 : b0;
          if (blk >= 0)
            tma_load_2d(smem + L::kOffCode + cs * 2 * kCodeTile + which * kCodeTile + (32 * lw + 16 * r) * 128,
                        which ? tmap_v : tmap_k, &cbar[cs], 0, (int32_t)(((int64_t)blk * p.num_kv_heads + g) * bs));
        }
        ++issued;
      };
      for (int j = 0; j < kCS && j < nkt; ++j) issue_codes(j);
      for (int j = 0; j < nkt && ok; ++j) {
        const int s = j % kStages, cs = j % kCS;
        const uint32_t ph_prev = ((j / kStages) - 1) & 1;
        if (!wait_slot(&cbar[cs], (j / kCS) & 1)) break;
        const uint8_t *cst = smem + L::kOffCode + cs * 2 * kCodeTile;
#pragma unroll
        for (int qi = 0; qi < 4; ++qi) {
          const int which = qi >> 1, r = qi & 1;
          if (r == 0 && j >= kStages && !wait_slot(which ? &v_free[s] : &k_free[s], ph_prev)) break;
          const int nval = (int)((nvs >> (16 * cs + 8 * r)) & 0xffu);   // rows past the sequence end: zeros
          uint8_t *tile = smem + (which ? L::kOffV : L::kOffK) + s * kTileBytes + pn * kTilePanel;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rr = 4 * i + (lane >> 3), row = 32 * lw + 16 * r + rr;
            const uint4 cw = rr < nval ? *reinterpret_cast<const uint4 *>(cst + which * kCodeTile + row * 128 +
                                                                            ((q ^ (row & 7)) << 4))
                                       : make_uint4(0, 0, 0, 0);
            uint32_t o[8];
            widen16<__half>(cw, o);   // the MMAs take f16 operands with an fp8 cache
            uint8_t *dst = tile + row * 128;
            *reinterpret_cast<uint4 *>(dst + ((c0 ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(dst + (((c0 + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          if (r == 1) {
            fence_async_smem();
            mbar_arrive(which ? &v_full[s] : &k_full[s]);
          }
        }
        if (!ok) break;
        // code stage cs is read: its next boxes (generic reads before the async-proxy writes)
        fence_async_smem();
        if (j + kCS < nkt) issue_codes(j + kCS);
      }
      // no box of this warp in flight at exit (bounded waits)
      for (int jj = max(0, issued - kCS); jj < issued; ++jj)
        wait_or_abort(&cbar[jj % kCS], (jj / kCS) & 1, p.err, abort_flag);
    } else {
      // fp8 rows (128 B), two Q tiles: per instruction 4 rows x 8 words of 16
      // codes.  A tile is four quarters (K run 0, K run 1, V run 0, V run 1).
      // The loads run kPf quarters (half a tile) ahead of the widening into
      // shared memory.
      constexpr int kPf = 2;
      const int q = lane & 7, pn = q >> 2, c0 = (2 * q) & 7;
      auto load = [&](int j, int qi, uint4 (&w)[4]) {
        int64_t row0;
        const int nval = rows_of(j, qi & 1, row0);
        const char *pool = (qi >> 1) ? vpool : kpool;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * i + (lane >> 3);
          w[i] = rr < nval ? ld_nc16(pool + (row0 + rr) * kRowBytes + q * 16) : make_uint4(0, 0, 0, 0);
        }
      };
      uint4 buf[kPf][4];   // quarter g of the load order in buf[g % kPf]
#pragma unroll
      for (int g = 0; g < kPf; ++g)
        if (g / 4 < nkt) load(g / 4, g % 4, buf[g]);
      for (int j = 0; j < nkt && ok; ++j) {
        const int s = j % kStages;
        const uint32_t ph_prev = ((j / kStages) - 1) & 1;
#pragma unroll
        for (int qi = 0; qi < 4; ++qi) {
          const int which = qi >> 1, r = qi & 1;
          if (r == 0 && j >= kStages && !wait_slot(which ? &v_free[s] : &k_free[s], ph_prev)) break;
          uint8_t *tile = smem + (which ? L::kOffV : L::kOffK) + s * kTileBytes + pn * kTilePanel;
          uint4 (&cur)[4] = buf[qi % kPf];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = 32 * lw + 16 * r + 4 * i + (lane >> 3);
            uint32_t o[8];
            widen16<__half>(cur[i], o);   // the MMAs take f16 operands with an fp8 cache
            uint8_t *dst = tile + row * 128;
            *reinterpret_cast<uint4 *>(dst + ((c0 ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(dst + (((c0 + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          // refill the buffer with the quarter kPf ahead in the load order
          const int g = 4 * j + qi + kPf;
          if (g / 4 < nkt) load(g / 4, g % 4, cur);
          if (r == 1) {
            fence_async_smem();
            mbar_arrive(which ? &v_full[s] : &k_full[s]);
          }
        }
      }
    }
    // before exit: the MMAs' releases of the last tiles have arrived, and no copy is in flight
    if (ok) {
      for (int tt = max(0, nkt - kStages); tt < nkt; ++tt) {
        wait_or_abort(&k_free[tt % kStages], (tt / kStages) & 1, p.err, abort_flag);
        wait_or_abort(&v_free[tt % kStages], (tt / kStages) & 1, p.err, abort_flag);
      }
    }
    if constexpr (!kFp8) cp_async_wait_all();
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issue (warp kMmaWarp; warps
    // past it, in a larger block such as the mixed launch's, have no role)
    // The whole warp runs the schedule (so descriptors stay warp-uniform); one
    // elected lane issues the MMAs and their commits.  Per key tile j and Q
    // tile t: O_t += P_t(j) V_j, then -- once that P.V is complete, because
    // the scores of tile j+1 go where P_t(j) is -- S_t(j+1) = Q_t K_{j+1}^T.
    const bool leader = elect_one();
    const uint32_t idesc_s = umma_idesc(kAB, kN, false);
    const uint32_t idesc_o = umma_idesc(kAB, kD, true);
    const uint64_t qdesc = umma_desc(smem_u32(smem + L::kOffQ), 16);
    const uint64_t kdesc0 = umma_desc(smem_u32(smem + L::kOffK), 16);
    const uint64_t vdesc0 = umma_desc(smem_u32(smem + L::kOffV), kTilePanel);
    auto wait_all = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p.err, abort_flag));
    };
    bool ok = nkt == 0 || wait_all(q_ready, 0);
    bool issued = false;
    auto issue_s = [&](int t, int j) {  // S_t(j) = Q_t K_j^T into buffer j % kBufs (K tile j waited for)
      const uint64_t kd = kdesc0 + (((j % kStages) * kTileBytes) >> 4);
      const uint64_t qd = qdesc + ((t * kQBytes) >> 4);
      const int bb = j % kBufs;
      if (leader) {
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          umma(sbuf(t, bb), qd + (((k >> 2) * (kM * 128) + (k & 3) * 32) >> 4),
               kd + (((k >> 2) * kTilePanel + (k & 3) * 32) >> 4), idesc_s, k > 0 ? 1u : 0u);
        umma_commit(&s_full[t * kBufs + bb]);
      }
      __syncwarp();
      issued = true;
    };
    // the first kBufs score tiles
    for (int jj = 0; jj < kBufs && jj < nkt && ok; ++jj) {
      ok = wait_all(&k_full[jj % kStages], (jj / kStages) & 1);
      if (!ok) break;
      fence_async_smem();
      tc_fence_after();
      for (int t = 0; t < kQTiles; ++t) issue_s(t, jj);
      if (leader) umma_commit(&k_free[jj % kStages]);
      __syncwarp();
    }
    for (int j = 0; j < nkt && ok; ++j) {
      const int s = j % kStages, b = j % kBufs;
      ok = wait_all(&v_full[s], (j / kStages) & 1);
      if (!ok) break;
      const int jn = j + kBufs;                 // the score tile that reuses buffer b
      const bool more = jn < nkt;
      const int sn = jn % kStages;
      const uint64_t vd = vdesc0 + ((s * kTileBytes) >> 4);
      for (int t = 0; t < kQTiles && ok; ++t) {
        ok = wait_all(&p_full[t * kBufs + b], (j / kBufs) & 1);
        if (!ok) break;
        fence_async_smem();   // V tile written through the generic proxy (cp.async / st.shared)
        tc_fence_after();
        if (leader) {
#pragma unroll
          for (int half = 0; half < (kSplit ? 2 : 1); ++half) {
#pragma unroll
            for (int kk = 0; kk < kN / 16; ++kk)   // keys 16kk..16kk+15: P hi at column 16kk, lo at 16kk+8
              umma_ts(obuf(t), sbuf(t, b) + 16 * kk + 8 * half, vd + ((kk * 16 * 128) >> 4), idesc_o,
                      (j > 0 || half > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&o_done[t]);
          if (t == kQTiles - 1) umma_commit(&v_free[s]);
        }
        __syncwarp();
        if (more) {
          if (t == 0) {
            ok = wait_all(&k_full[sn], (jn / kStages) & 1);
            if (!ok) break;
          }
          // S_t(jn) overwrites P_t(j): wait for its P.V
          ok = wait_all(&o_done[t], j & 1);
          if (!ok) break;
          fence_async_smem();
          tc_fence_after();
          issue_s(t, jn);
          if (t == kQTiles - 1 && leader) umma_commit(&k_free[sn]);
          __syncwarp();
        }
      }
    }
    // every MMA issued above is complete before tensor memory is freed
    if (issued) {
      if (leader) umma_commit(fin);
      __syncwarp();
      mbar_wait(fin, 0, p.err);
    }
  }

  // ===================================================== teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
  }
}

template <typename KV, typename QT, int G, int kQTiles>
__global__ void __launch_bounds__(tc::Roles<kQTiles>::kThreads, 1)
    prefill_tc_kernel(const PrefillTcParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  prefill_tc_body<KV, QT, G, kQTiles>(p, blockIdx.x, blockIdx.y, &tmap_k, &tmap_v);
}

// Host launcher: grid (chunks x row blocks, KV heads), one CTA per SM.  Two Q
// tiles per CTA share every K/V tile, unless that leaves SMs idle (few rows):
// then one Q tile per CTA doubles the grid.
template <typename KV, typename QT, int G, int kQTiles>
cudaError_t launch_prefill_tc_tiles(const PrefillTcParams &p0, const PoolMaps &m, int num_chunks, cudaStream_t s) {
  constexpr int smem = tc::Layout<kQTiles, std::is_same<KV, uint8_t>::value>::kSmemBytes;
  constexpr int BR = kQTiles * tc::kM / G;
  PrefillTcParams p = p0;
  p.row_blocks = (p.max_q_len + BR - 1) / BR;
  auto kern = prefill_tc_kernel<KV, QT, G, kQTiles>;
  cudaError_t e = ensure_smem_limit<prefill_tc_kernel<KV, QT, G, kQTiles>>(smem);
  if (e != cudaSuccess) return e;
  const int64_t gx = (int64_t)num_chunks * p.row_blocks;
  if (gx > 2147483647ll || p.num_kv_heads > 65535) return cudaErrorInvalidValue;
  dim3 grid((unsigned)gx, (unsigned)p.num_kv_heads);
  kern<<<grid, tc::Roles<kQTiles>::kThreads, smem, s>>>(p, m.k, m.v);
  return cudaGetLastError();
}

template <typename KV, typename QT, int G>
cudaError_t launch_prefill_tc_one(const PrefillTcParams &p, const PoolMaps &m, int num_chunks, int num_sms,
                                  cudaStream_t s) {
  const int64_t two = (int64_t)num_chunks * ((p.max_q_len + 2 * tc::kM / G - 1) / (2 * tc::kM / G)) * p.num_kv_heads;
  if (two >= num_sms) return launch_prefill_tc_tiles<KV, QT, G, 2>(p, m, num_chunks, s);
  return launch_prefill_tc_tiles<KV, QT, G, 1>(p, m, num_chunks, s);
}

// m: with an fp8 cache, each pool as [rows][128 codes] with one cache block per
// box (encode_pool_map_fp8_blocks); unused with a 16-bit cache.
template <typename KV, typename QT>
cudaError_t launch_prefill_tc(const PrefillTcParams &p, const PoolMaps &m, int gqa, int num_chunks, cudaStream_t s) {
  int num_sms = 0;
  if (current_sm_count(&num_sms) != cudaSuccess) return cudaErrorUnknown;
  switch (gqa) {
    case 1: return launch_prefill_tc_one<KV, QT, 1>(p, m, num_chunks, num_sms, s);
    case 2: return launch_prefill_tc_one<KV, QT, 2>(p, m, num_chunks, num_sms, s);
    case 4: return launch_prefill_tc_one<KV, QT, 4>(p, m, num_chunks, num_sms, s);
    case 8: return launch_prefill_tc_one<KV, QT, 8>(p, m, num_chunks, num_sms, s);
    case 16: return launch_prefill_tc_one<KV, QT, 16>(p, m, num_chunks, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
