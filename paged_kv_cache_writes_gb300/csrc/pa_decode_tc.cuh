// pa_decode_tc.cuh -- paged decode for grouped-query attention on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory),
// G = 4, 8 or 16 query rows per KV head (other groups padded), head_dim 128
// with G up to 16 or head_dim 64 with G up to 8, any cache dtype.
//
// What it computes: the same as the CUDA-core decode (pa_decode.cuh).  For
// each sequence and query head h,
//   out[row][h] = sum_p softmax_p(scale * q[row][h] . K[p][g]) V[p][g],
// g the KV head of h, K/V gathered through the block table ("Inside vLLM
// Architecture", sections "Architectural Anatomy: PagedAttention Virtual
// Memory Paging" and "CUDA Shared Memory Optimization in PagedAttention").
// A row is cut into partitions of at most 512 tokens whose partial results
// are merged by their log-sum-exp, as in the CUDA-core kernel, by a warp of
// the CTA whose softmax warps wrote the row's last partition.  The merge and
// the counting of finished partitions stay off the softmax warps' path: they
// are one stage of the CTA's pipeline, and waiting there on dependent global
// reads stalled every other stage (measured: merging inline took more than
// half of their time).
//
// Why tensor cores.  The G query heads of a KV head all read every K and V
// element: G multiply-adds per K element and G per V element.  With a bf16
// cache and G = 8 that is 4 fp32 FMAs per byte of cache, about 27 T FMA/s at
// the GPU's copy bandwidth, two thirds of the CUDA cores' fp32 rate before any
// conversion or softmax work (measured: the CUDA-core kernel takes the same
// time on an fp8 cache as on a bf16 one, so it is not bound by memory).  Per
// (sequence, KV head) the work is a dense [G x 128] x [128 x keys] product
// and its [G x keys] x [keys x 128] partner: the contraction of prefill with
// G query rows.
//
// Transposed tiles.  With only G query rows the keys take the MMA's M side:
//   S^T (128 keys x 16)  = K_tile (128 x 128, K-major) . Q^T (K-major: the q rows)
//   O^T (128 d x N_O)   += V_tile^T (MN-major view of the tile as stored) . P^T
// S^T lands in tensor memory with lane = key, column = head; O^T with lane =
// head element d, column = head.  Q rows G..15 are zero.  With head_dim 64 a
// row is one 128-byte panel; O^T keeps M = 128 with both 64-element halves of
// its A operand read from that one panel, so lanes 64..127 repeat lanes 0..63
// and are ignored.  P^T is staged in
// shared memory (K-major, lane = key writes its column): columns 0..G-1 hold
// p (its bf16 hi part for a bf16 cache) and, for a bf16 cache, columns
// G..2G-1 hold the lo part p - hi, so one MMA per 16 keys accumulates both
// and the epilogue adds the two halves of O^T.
//
// fp8 caches: the e4m3 codes are the MMA operands as stored (kind::f8f6f4,
// 32 keys or elements per MMA), so a tile goes from the bulk copy to the
// MMAs untouched.  The other operand is then e4m3 too, as a sum of terms:
// 256 p is written as hi + lo / 16 (hi in rows 0..G-1 of P^T, lo in rows
// G..2G-1), which holds it to 2^-8 of itself; the query rows, scaled by a
// power of two 2^e per unit (|q| 2^e in [128, 256) at the unit's largest
// element), likewise as hi + lo / 16 for bf16 queries and as hi + mid / 16 +
// lo / 256 in rows 0..3G-1 for f16 queries: either holds every query element
// within 2^-13 of the unit's largest exactly (8 or 11 significant bits).  The
// softmax and the epilogue add the column groups of S^T and O^T and undo the
// scales.
//
// Softmax per unit (no online rescale): all tiles of a unit (<= 4 x 128
// keys) are scored first, the exact maximum per head over the unit comes from
// a warp reduction and one exchange between the four softmax warps (an
// mbarrier, bounded), then p = 2^(t - max) for every key.  The exchange also
// carries the previous unit's row sums, which its epilogue needs.
//
// Work: a unit is (row, partition, KV head), listed by a plan kernel (rows
// with the most partitions first, each row's partitions together) and
// claimed from an atomic cursor by a persistent CTA per SM.  Roles:
//  * warps 0-3, softmax and epilogue: thread i owns tensor-memory lane i (key
//    i of a score tile, element d = i of an output row);
//  * loader warps (NL of them): the ring's tiles, in the MMAs' order (K
//    tiles of unit u, then V tiles of unit u-1), go to the loaders in turn by
//    ring position; each tile is one bulk-tensor copy per cache block
//    straight into its slot in the MMA's 128-byte-swizzled layout (32 KB for
//    a 16-bit cache, 16 KB for fp8).  Loader 0 also stages Q^T (16-bit
//    caches, cp.async).  One warp issuing the copies of 4 KB blocks one
//    after another streamed at most ~21 bytes per SM clock, so the decode
//    and mixed launches have four loaders (one with 16 query heads per KV
//    head, whose softmax needs more registers than nine or more warps leave);
//  * MMA warp (one elected lane issues): S^T of unit u, then O^T of unit
//    u-1, whose softmax ran while the scores of u were computed;
//  * scheduler warp: claims units (two at a time with fp8, else one) and publishes each, with
//    the block ids of its tiles, in a ring of six descriptors, so the chain
//    of dependent reads behind a claim (cursor, work item, sequence length,
//    block table) runs ahead of the loads instead of between them.  It also
//    stores a fused step's new token (pa_decode_write) before publishing the
//    unit that reads it, and with an fp8 cache writes the unit's Q^T (the
//    query rows' scale and two e4m3 terms) beside the descriptor, so that no
//    dependent global read stalls the loader;
//  * merge warp: merges split rows taken from a grid-wide list that the
//    softmax warps append to, so the merging is shared by every CTA.
//
// Every mbarrier wait is bounded (PA_ERR_TIMEOUT, after which the CTA
// abandons its work); tensor memory is freed only after every issued MMA has
// completed.
#pragma once

#include <type_traits>

#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

// A split row (sequence, KV head) whose partitions are all written, in the
// workspace's merge list: one 64-bit word, row << 32 | kvh << 13 | nparts,
// stored with release once the partials are published and read with one
// acquire load (nparts >= 2, so a published word is never 0; the plan kernel
// zeroes the list).  The merge needs no second round trip for the record.
struct DecodeMergeJob {
  uint64_t word;
  uint64_t unused;   // 16-byte records
};
__device__ __forceinline__ uint64_t merge_word(int row, int kvh, int nparts) {
  return ((uint64_t)(uint32_t)row << 32) | ((uint64_t)(uint32_t)kvh << 13) | (uint64_t)(uint32_t)nparts;
}

struct DecodeTcParams {
  DecodeParams d;            // shapes, plan and workspace (d.groups = 1: a unit serves all G heads)
  DecodeMergeJob *jobs;      // merge list, one record per split (row, KV head); d.hdr->pad[0..2]:
                             // records appended, records claimed, records in all
  const void *k_cache;       // [num_blocks][Hkv][block_size][128]
  const void *v_cache;
  float s_mult;              // scale * log2(e) (* k_scale for an fp8 cache); any sign
  // Fused cache write (pa_decode_write), or k_new == nullptr: row i's new token
  // k_new/v_new[i] ([Hkv][128] in the query dtype, rows new_stride elements
  // apart) goes to slot new_slots[i] (negative: none), which must be the slot of
  // position seq_lens[i] - 1; fp8 caches store e4m3(fp32(x) / scale).
  const void *k_new;
  const void *v_new;
  int64_t new_stride;
  const int64_t *new_slots;
  float k_scale, v_scale;
};

namespace dtc {

constexpr int kD = 128;                   // head_dim
constexpr int kKeys = 128;                // keys per tile (MMA M, tensor-memory lanes)
constexpr int kMaxTiles = 4;              // tiles per unit: partitions hold <= 512 tokens
constexpr int kInfo = 6;                  // unit descriptors in flight (bounds how far a CTA claims ahead)
constexpr int kClaimMax = 2;              // units per claim at most (claims are 1 or 2 units)
constexpr int kRep = 8;                   // split units handed from the softmax warps to the merge warp
// A 16-bit K or V tile in shared memory: 16 atoms of 8 keys, atom a at
// a * 2048, its first 64 elements (128-byte rows, 128-byte swizzle) at +0 and
// the last 64 at +1024 -- the layout of a 4D bulk-tensor box {64, 8 rows,
// 2 panels, block_size / 8 atoms} over one cache block.
constexpr int kAtomBytes = 2048;          // 8 keys x 256 B: the two 128-byte panels of 8 rows

// Warp roles: 0-3 softmax, 4 the loader (bulk-tensor copies and Q), 5 the
// MMA warp, 6 the scheduler, 7 the merge warp.
struct Roles {
  static constexpr int kLoadWarp = 4;    // loader 0 (also stages Q^T)
  static constexpr int kMmaWarp = 5;
  static constexpr int kSchedWarp = 6;
  static constexpr int kMergeWarp = 7;
  static constexpr int kLoadWarp1 = 8;   // loaders 1 .. NL-1, then (kSepMerge) the merging warp
  // Loader warps of the decode launch, and whether a separate warp merges the
  // split rows (the merge warp then only counts its CTA's reports): nine to
  // twelve warps leave 168 registers per thread (three warps on one of the
  // SM's four register files), too few for the softmax of 16 heads, which
  // keeps one loader and one merge warp.
  static constexpr int loaders(int g) { return g <= 8 ? 4 : 1; }
  static constexpr bool sep_merge(int g) { return g <= 8; }
  static constexpr int merge2_warp(int nl) { return kLoadWarp1 + nl - 1; }
  static constexpr int threads_for(int nl, bool sep = false) {
    return (kLoadWarp1 + (nl > 1 ? nl - 1 : 0) + (sep ? 1 : 0)) * 32;
  }
};

constexpr int kMaxSlots = 12;

// A claimed unit as published by the scheduler warp: its place, and the
// block id of each 16-key run of its tiles (run r of tile j at blk[8*j + r];
// -1 past the end of the unit).  qscale: fp8 caches, the bits of the power
// of two its query rows are multiplied by before their e4m3 split.
struct TcUnit {
  int32_t valid, row, kvh, part, tok_begin, ntok, nparts, qscale;
  int32_t blk[kMaxTiles * 8];
};

// e4m3 terms per query value with an fp8 cache: two hold a bf16 value's 8
// significant bits, three an f16 value's 11; 1 (no split) for 16-bit caches.
template <typename KV, typename QT>
struct QTerms {
  static constexpr int value = !std::is_same<KV, uint8_t>::value ? 1 : std::is_same<QT, __half>::value ? 3 : 2;
};

// Shared-memory and tensor-memory geometry.  16-bit caches: K/V tiles of
// 32 KB (two 128-byte panels per 8-key atom), Q^T of 16 rows (the heads,
// padded) and P^T of kNO rows, each in two 64-element panels.  fp8 caches:
// tiles of 128 rows of head_dim codes (16 KB with the 128-byte swizzle, or 8
// KB of 64-byte rows with the 64-byte swizzle for head_dim 64: the layouts a
// 2D bulk-tensor box writes), Q^T of head_dim-byte rows in the same swizzle
// and P^T of one 128-key panel, holding the hi terms in rows 0..G-1, the lo
// terms in rows G..2G-1 (and with three query terms, the last in rows
// 2G..3G-1 of Q^T).
template <int G, bool kSplit, bool kFp8, int kQTerms = 1, int D = 128>
struct TcGeo {
  static_assert(G == 4 || G == 8 || G == 16, "4, 8 or 16 query heads per KV head");
  static_assert(D == 128 || D == 64, "head_dim 128 or 64");
  static constexpr int kPanels = D / 64;                            // 128-byte panels of a 16-bit row
  static constexpr int kAtom = 8 * 2 * D;                           // 8 keys of a 16-bit tile (all panels)
  static constexpr int kPRows = (kSplit || kFp8) ? 2 * G : G;       // P^T rows in use
  static constexpr int kNO = kPRows <= 16 ? 16 : 32;                // O^T columns (MMA N)
  static constexpr int kQRows = kQTerms * G;                        // Q^T rows in use
  static constexpr int kNS = kQRows <= 16 ? 16 : (kQRows + 15) / 16 * 16;   // S^T columns per tile (MMA N)
  static constexpr int kSCols = kFp8 ? kNS : G;                     // S^T columns read per tile
  static constexpr int kQBytes = kFp8 ? kNS * D : kPanels * kNS * 128;    // Q^T of a unit
  // Q^T buffers: fp8, one per unit descriptor (written by the scheduler warp
  // with the descriptor); 16-bit, two (copied by the loader per unit parity)
  static constexpr int kQBufs = kFp8 ? kInfo : 2;
  static constexpr int kPBytes = kFp8 ? kNO * 128 : 2 * kNO * 128;  // P^T of a tile
  static constexpr int kSlotBytes = kFp8 ? kKeys * D : kKeys * D * 2;     // one K or V tile
  static constexpr int kColO = 2 * kMaxTiles * kNS;                 // tensor-memory column of O^T, buffer 0
  static constexpr int kTmemCols = kColO + 2 * kNO <= 256 ? 256 : 512;
  static constexpr int kNumBars = 2 * kMaxSlots + 8 * 2 + 2 * kInfo + 1 + 2 * kRep;
  static constexpr int kOffQ = 0;                                        // [kQBufs] Q^T
  static constexpr int kOffP = kOffQ + kQBufs * kQBytes;                 // [2][4] P^T
  static constexpr int kOffRed = kOffP + 2 * kMaxTiles * kPBytes;        // float [2][4 warps][2][16]
  static constexpr int kOffInfo = kOffRed + 2 * 4 * 2 * 16 * 4;          // TcUnit [kInfo] (16-byte aligned)
  static constexpr int kOffBar = kOffInfo + kInfo * (int)sizeof(TcUnit);
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRep = (kOffMisc + 16 + 15) / 16 * 16;         // int4 [kRep] reports (16-byte aligned)
  static constexpr int kOffRing = (kOffRep + kRep * 16 + 1023) / 1024 * 1024;  // [kSlots] K/V tiles
  static constexpr int kSlots0 = (227 * 1024 - 1024 - kOffRing) / kSlotBytes;
  static constexpr int kSlots = kSlots0 > kMaxSlots ? kMaxSlots : kSlots0;
  static constexpr int kSmemBytes = kOffRing + kSlots * kSlotBytes + 1024;  // + alignment slack
  static_assert(kSlots >= 2 && kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kOffRep % 16 == 0 && kOffInfo % 16 == 0 && kOffBar % 8 == 0 && kOffMisc % 8 == 0,
                "aligned reports, descriptors and barriers");
  static_assert(kOffRing % 1024 == 0 && kOffP % 1024 == 0 && kQBytes % 1024 == 0 && kPBytes % 1024 == 0,
                "1024-byte swizzle atoms");
};

// N consecutive fp32 columns of this thread's tensor-memory lane (warp-collective).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 4) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
  } else if constexpr (N == 8) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
  } else if constexpr (N == 16) {
    tc::tmem_ld16(taddr, v);
  } else if constexpr (N == 32) {
    tc::tmem_ld32(taddr, v);
  } else {
    static_assert(N == 48, "4, 8, 16, 32 or 48 columns");
    float a[32], b[16];
    tc::tmem_ld32(taddr, a);
    tc::tmem_ld16(taddr + 32, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = a[i];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[32 + i] = b[i];
  }
}

// Reduce v[h] (h < G) over the 32 lanes of the warp by halving exchanges:
// each level swaps half of the remaining heads with the partner lane.  The
// lane ends with the reduction of head lane >> (5 - log2 G).
template <int G, bool kMax>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[G], int lane) {
  constexpr int kLog = G == 4 ? 2 : G == 8 ? 3 : 4;
#pragma unroll
  for (int lv = 0; lv < kLog; ++lv) {
    const int n = G >> lv, mask = 16 >> lv;
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? v[k] : v[k + n / 2];
      const float keep = upper ? v[k + n / 2] : v[k];
      const float got = __shfl_xor_sync(0xffffffffu, send, mask);
      v[k] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int mask = 16 >> kLog; mask > 0; mask >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], mask);
    v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

// The descriptor's header, copied to registers (the block ids stay in shared memory).
struct UnitHdr {
  int32_t valid, row, kvh, part, tok_begin, ntok, nparts, qscale;
};
__device__ __forceinline__ UnitHdr read_unit(const TcUnit *u) {
  const volatile int32_t *s = reinterpret_cast<const volatile int32_t *>(u);
  UnitHdr r;
  r.valid = s[0];
  r.row = s[1];
  r.kvh = s[2];
  r.part = s[3];
  r.tok_begin = s[4];
  r.ntok = s[5];
  r.nparts = s[6];
  r.qscale = s[7];
  return r;
}

__device__ __forceinline__ int num_tiles(const UnitHdr &u) { return u.valid ? (u.ntok + kKeys - 1) / kKeys : 0; }

// Largest |x| of the 8 query elements in a 16-byte word (NaN ignored).
__device__ __forceinline__ float absmax8(uint4 w, __nv_bfloat16) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(__uint_as_float((ws[i] << 16) & 0x7fffffffu),
                                                 __uint_as_float(ws[i] & 0x7fff0000u)));
  return m;
}
__device__ __forceinline__ float absmax8(uint4 w, __half) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&ws[i]));
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

// The power of two 2^e with amax * 2^e in [128, 256) (e clamped to +-100;
// 1 for amax = 0), as fp32 bits.
__device__ __forceinline__ int32_t query_scale_bits(float amax) {
  const int eb = (int)((__float_as_uint(amax) >> 23) & 0xff);
  const int e = amax > 0.f ? max(-100, min(100, 134 - eb)) : 0;
  return (e + 127) << 23;
}

}  // namespace dtc

// The decode CTA, for decode_tc_kernel and for the decode CTAs of the mixed
// kernel (pa_mixed_tc.cuh).  Warps past the eight roles (a wider mixed block)
// only take part in the two CTA-wide barriers.
template <typename KV, typename QT, int G, int D = 128, int NL = 1, bool kSepMerge = false, bool kPadRows = false>
__device__ __forceinline__ void decode_tc_body(const DecodeTcParams &tp, const CUtensorMap *tmap_k,
                                               const CUtensorMap *tmap_v) {
  using namespace tc;
  using namespace dtc;
  constexpr int kD = D;                       // head_dim (hides dtc::kD)
  constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  constexpr int kLoadWarp = Roles::kLoadWarp, kMmaWarp = Roles::kMmaWarp;
  constexpr int kSchedWarp = Roles::kSchedWarp, kMergeWarp = Roles::kMergeWarp;
  constexpr int kThreads = Roles::threads_for(NL, kSepMerge), kLoadWarp1 = Roles::kLoadWarp1;
  constexpr int kMerge2Warp = Roles::merge2_warp(NL);   // with kSepMerge: merges only
  // MMA operands: the cache's type (bf16 / f16 with a 16-bit cache, the queries
  // in the same type; e4m3 with an fp8 cache, the queries and P as two e4m3 terms)
  constexpr bool kBf16 = std::is_same<QT, __nv_bfloat16>::value && !kFp8;
  constexpr bool kSplit = kBf16;            // bf16 cache: P as hi + lo
  constexpr int kQTerms = QTerms<KV, QT>::value;
  using GE = TcGeo<G, kSplit, kFp8, kQTerms, D>;
  // The MMA warp consumes the ring in order, so a loader's wait for the consumption of
  // position g - S is never two phases behind while it has NL <= S positions in hand.
  static_assert(GE::kSlots >= NL, "at least as many ring slots as loaders (parity waits stay within one phase)");
  constexpr int kAtomB = GE::kAtom;           // bytes of 8 keys of a 16-bit tile
  constexpr int kRowChunks = kD * 2 / 16;     // 16-byte chunks of a 16-bit row
  constexpr int S = GE::kSlots, kNO = GE::kNO, kNS = GE::kNS;
  constexpr uint32_t kAB = kBf16 ? 1u : 0u;   // instruction-descriptor format: bf16 1, f16 0, e4m3 0
  const DecodeParams &p = tp.d;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + GE::kOffBar);
  uint64_t *slot_full = bars;                 // [S] tile staged
  uint64_t *slot_free = bars + kMaxSlots;     // [S] the MMAs reading the tile are complete
  uint64_t *q_full = bars + 2 * kMaxSlots;    // [2] Q^T of unit buffer b staged (every loader thread)
  uint64_t *q_free = q_full + 2;              // [2] its S^T MMAs are complete
  uint64_t *s_full = q_free + 2;              // [2] S^T of every tile of the unit ready
  uint64_t *s_free = s_full + 2;              // [2] read by every softmax thread (128)
  uint64_t *p_full = s_free + 2;              // [2] P^T written (128)
  uint64_t *o_full = p_full + 2;              // [2] O^T complete
  uint64_t *o_free = o_full + 2;              // [2] O^T read by every softmax thread (128)
  uint64_t *red_bar = o_free + 2;             // [2] per-warp maxima and sums exchanged (128)
  uint64_t *info_full = red_bar + 2;          // [kInfo] unit descriptor published (32 scheduler lanes)
  uint64_t *info_free = info_full + kInfo;    // [kInfo] released by the MMA warp, the softmax warps and every loader
  uint64_t *fin = info_free + kInfo;          // every MMA of the CTA complete
  uint64_t *rep_full = fin + 1;               // [kRep] a split unit's partials stored (one arrival per softmax warp)
  uint64_t *rep_free = rep_full + kRep;       // [kRep] its report taken by the merge warp
  TcUnit *info = reinterpret_cast<TcUnit *>(smem + GE::kOffInfo);
  float *red = reinterpret_cast<float *>(smem + GE::kOffRed);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + GE::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + GE::kOffMisc + 8);
  // [kRep] reports {row, KV head, partitions (-1: the softmax warps are done), 0}; ordered
  // by the report barriers
  int4 *reports = reinterpret_cast<int4 *>(smem + GE::kOffRep);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Q^T and P^T buffers start zeroed: their padding rows are never written
  for (int i = tid; i < (GE::kOffRed - GE::kOffQ) / 16; i += kThreads)   // (threads past kThreads repeat zeros)
    reinterpret_cast<uint4 *>(smem + GE::kOffQ)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&slot_full[s], 1);   // one expect-tx arrival
      mbar_init(&slot_free[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_full[b], 32);     // every loader lane
      mbar_init(&q_free[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 128);
      mbar_init(&p_full[b], 128);
      mbar_init(&o_full[b], 1);
      mbar_init(&o_free[b], 128);
      mbar_init(&red_bar[b], 128);
    }
    for (int i = 0; i < kInfo; ++i) {
      mbar_init(&info_full[i], 32);   // every scheduler lane, after its own stores
      mbar_init(&info_free[i], 2 + NL);   // O^T issued, epilogue done, each loader past the unit
    }
    mbar_init(fin, 1);
    for (int i = 0; i < kRep; ++i) {
      mbar_init(&rep_full[i], 4);   // lane 0 of each softmax warp, after the warp's stores
      mbar_init(&rep_free[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensor_map(tmap_k);
    prefetch_tensor_map(tmap_v);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(GE::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_async_smem();   // the zeroed operand rows, for the MMAs' reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // launched as the plan kernel's programmatic dependent: everything above overlapped it;
  // its work list, cursor and counters are complete and visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next step's plan kernel may launch (it waits for this grid before it starts its work)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  auto col_s = [&](int b, int j) { return tmem + (uint32_t)((b * kMaxTiles + j) * kNS); };
  auto col_o = [&](int b) { return tmem + (uint32_t)(GE::kColO + b * kNO); };
  auto wait_all = [&](uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_or_abort(bar, parity, p.err, abort_flag));
  };

  const int hkv = p.num_kv_heads;
  const int hq = p.num_q_heads;
  // query heads per KV head: G, or with kPadRows 1..G, a unit's rows gr..G-1 then being
  // padding, with q = 0 (finite scores and softmax), never read from or written to global memory
  const int gr = kPadRows ? hq / hkv : G;

  // Merge the split row of record t of the grid-wide merge list (its ready flag
  // acquired by lane 0): out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p
  // over the row's partitions p (m_p in log2 units, M their maximum), kept as a
  // running maximum; lane l merges elements 4l..4l+3 of all G heads, the loads
  // of two partitions for every head in flight together.
  auto merge_job = [&](uint64_t word) {   // the record as lane 0 acquired it
    word = ((uint64_t)__shfl_sync(0xffffffffu, (uint32_t)(word >> 32), 0) << 32) |
           __shfl_sync(0xffffffffu, (uint32_t)word, 0);
    const int job_row = (int)(word >> 32), job_kvh = (int)((word >> 13) & 0x7ffffu), job_np = (int)(word & 0x1fffu);
    __syncwarp();   // lane 0's acquire of the record orders every lane's reads of the partials
    const int64_t head0 = (int64_t)job_row * hq + (int64_t)job_kvh * gr;
    float m[G], l[G];
    float4 acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = kNegInf;
      l[h] = 0.f;
      acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // two partitions per step: the loads of both are in flight together
    for (int q0 = 0; q0 < job_np; q0 += 2) {
      float2 ml[2][G];
      float4 a[2][G];
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const int q = min(q0 + k, job_np - 1);   // a lone last partition is read twice, merged once
          const int64_t e = (head0 + min(h, gr - 1)) * p.max_partitions + q;   // padding rows: a real head, unused
          ml[k][h] = __ldcg(&p.ws_ml[e]);
          a[k][h] = 4 * lane < kD ? __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + e * kD) + lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (q0 + k >= job_np) break;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(m[h], ml[k][h].x);
          const float so = fast_exp2(m[h] - mn), sn = fast_exp2(ml[k][h].x - mn);
          m[h] = mn;
          l[h] = l[h] * so + ml[k][h].y * sn;
          acc[h] = make_float4(acc[h].x * so + a[k][h].x * sn, acc[h].y * so + a[k][h].y * sn,
                               acc[h].z * so + a[k][h].z * sn, acc[h].w * so + a[k][h].w * sn);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float om = p.v_hs ? p.out_mult * __ldg(p.v_hs + job_kvh) : p.out_mult;
      const float inv = l[h] > 0.f ? om / l[h] : 0.f;
      const int64_t o0 = (head0 + h) * kD + 4 * lane;
      if (4 * lane >= kD || h >= gr) continue;   // head_dim 64: lanes 0..15; padding rows
      store_out<QT>(p.out, o0, p.out_f32 != 0, acc[h].x * inv);
      store_out<QT>(p.out, o0 + 1, p.out_f32 != 0, acc[h].y * inv);
      store_out<QT>(p.out, o0 + 2, p.out_f32 != 0, acc[h].z * inv);
      store_out<QT>(p.out, o0 + 3, p.out_f32 != 0, acc[h].w * inv);
    }
  };
  // Claim records of the merge list and merge them until every one is claimed:
  // the warps that have finished their own role help drain the list at the end
  // of the kernel.  Waiting for a claimed record is bounded (PA_ERR_TIMEOUT).
  auto drain = [&]() {
    const int total_jobs = __ldcg(&p.hdr->pad[2]);
    for (;;) {
      if (*abort_flag) return;
      int t = 0;
      if (lane == 0) t = atomicAdd(&p.hdr->pad[1], 1);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t >= total_jobs) return;
      uint64_t word = 0;
      if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        for (;;) {
          asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(word) : "l"(&tp.jobs[t].word) : "memory");
          if (word || *abort_flag) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            record_error(p.err, PA_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          __nanosleep(128);   // a short poll: the record's merge is on the kernel's tail
        }
      }
      if (!__shfl_sync(0xffffffffu, word != 0, 0)) return;
      merge_job(word);
    }
  };

  if (warp < kLoadWarp) {
    // ===================================================== softmax and epilogue (warps 0-3)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float c0 = tp.s_mult;
    constexpr int kLog = G == 4 ? 2 : G == 8 ? 3 : 4;
    const int my_head = lane >> (5 - kLog);
    const bool red_writer = (lane & ((1 << (5 - kLog)) - 1)) == 0;
    float l_part[G], m_prev[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l_part[h] = 0.f;
      m_prev[h] = kNegInf;
    }
    UnitHdr prev;
    prev.valid = 0;
    bool ok = true;
    // A split unit's partial results, once stored by every softmax warp, are
    // handed to the CTA's merge warp through a ring of reports (each warp arrives
    // after its stores); the merge warp publishes them to the rest of the GPU,
    // so that the release and its wait stay off the softmax warps' path.
    int n_rep = 0;
    auto hand_over = [&](int row, int kvh, int np) {   // np -1: no more reports
      const int rs = n_rep % kRep;
      if (n_rep >= kRep && !wait_all(&rep_free[rs], ((n_rep / kRep) - 1) & 1)) return false;
      if (tid == 0) reports[rs] = make_int4(row, kvh, np, 0);
      __syncwarp();   // the warp's stores precede lane 0's arrival
      if (lane == 0) mbar_arrive(&rep_full[rs]);
      ++n_rep;
      return true;
    };
    for (int u = 0; ok; ++u) {
      const int ib = u % kInfo, b = u & 1;
      ok = wait_all(&info_full[ib], (u / kInfo) & 1);
      if (!ok) break;
      const UnitHdr cur = read_unit(&info[ib]);
      const int nt = num_tiles(cur);
      float c = p.k_hs && cur.valid ? c0 * __ldg(p.k_hs + cur.kvh) : c0;
      if constexpr (kFp8) c *= __frcp_rn(__int_as_float(cur.valid ? cur.qscale : 127 << 23));   // exact: 2^-e
      // scores of this unit in log2 units, t = s * scale * log2(e); masked keys -inf
      float t[kMaxTiles][G];
      float mloc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) mloc[h] = kNegInf;
      if (cur.valid) {
        ok = wait_all(&s_full[b], (u >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kMaxTiles; ++j) {
          if (j < nt) {
            float raw[GE::kSCols];
            tmem_ld_cols<GE::kSCols>(col_s(b, j) + lane_base, raw);
            const bool kv = j * kKeys + tid < cur.ntok;
#pragma unroll
            for (int h = 0; h < G; ++h) {
              // fp8: hi + lo / 16, or hi + (mid + lo / 16) / 16
              const float sv = kQTerms == 3   ? fmaf(fmaf(raw[2 * G + h], 0.0625f, raw[G + h]), 0.0625f, raw[h])
                               : kQTerms == 2 ? fmaf(raw[G + h], 0.0625f, raw[h])
                                              : raw[h];
              t[j][h] = kv ? sv * c : kNegInf;
              mloc[h] = fmaxf(mloc[h], t[j][h]);
            }
          } else {
#pragma unroll
            for (int h = 0; h < G; ++h) t[j][h] = kNegInf;
          }
        }
        tc_fence_before();
        mbar_arrive(&s_free[b]);
      }
      // exchange: this unit's per-warp maxima and the previous unit's per-warp sums
      {
        const float wm = warp_reduce_heads<G, true>(mloc, lane);
        const float ws = warp_reduce_heads<G, false>(l_part, lane);
        float *rb = red + (b * 4 + warp) * 32;
        if (red_writer) {
          rb[my_head] = wm;
          rb[16 + my_head] = ws;
        }
        mbar_arrive(&red_bar[b]);
        ok = wait_all(&red_bar[b], (u >> 1) & 1);
        if (!ok) break;
      }
      float m_cur[G], l_prev[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float *r0 = red + (b * 4) * 32;
        m_cur[h] = fmaxf(fmaxf(r0[h], r0[32 + h]), fmaxf(r0[64 + h], r0[96 + h]));
        l_prev[h] = (r0[16 + h] + r0[48 + h]) + (r0[80 + h] + r0[112 + h]);
      }
      // P^T of this unit (its buffer's previous reader, P.V of unit u-2, finished
      // before the epilogue of u-2, which ran in the previous iteration)
      if (cur.valid && kFp8) {
        // 256 p = hi + lo / 16 in e4m3, key tid's byte of rows h and G + h
#pragma unroll
        for (int h = 0; h < G; ++h) l_part[h] = 0.f;
        uint8_t *pb = smem + GE::kOffP + b * kMaxTiles * GE::kPBytes + (tid & 15);
#pragma unroll
        for (int j = 0; j < kMaxTiles; ++j) {
          if (j >= nt) break;
          uint8_t *pt = pb + j * GE::kPBytes;
#pragma unroll
          for (int h = 0; h < G; h += 2) {
            const float msub0 = m_cur[h] == kNegInf ? 0.f : m_cur[h];
            const float msub1 = m_cur[h + 1] == kNegInf ? 0.f : m_cur[h + 1];
            const float p0 = fast_exp2(t[j][h] - msub0), p1 = fast_exp2(t[j][h + 1] - msub1);
            uint32_t hi, lo;
            split2_e4m3(make_float2(p0 * 256.f, p1 * 256.f), hi, lo);
            auto put = [&](int row, uint32_t code) { pt[row * 128 + (((tid >> 4) ^ (row & 7)) << 4)] = (uint8_t)code; };
            put(h, hi);
            put(h + 1, hi >> 8);
            put(G + h, lo);
            put(G + h + 1, lo >> 8);
            l_part[h] += p0;
            l_part[h + 1] += p1;
          }
        }
        fence_async_smem();
        mbar_arrive(&p_full[b]);
      } else if (cur.valid) {
#pragma unroll
        for (int h = 0; h < G; ++h) l_part[h] = 0.f;
        uint8_t *pb = smem + GE::kOffP + b * kMaxTiles * GE::kPBytes + (tid >> 6) * (kNO * 128) + (tid & 7) * 2;
        const int ck = (tid & 63) >> 3;
#pragma unroll
        for (int j = 0; j < kMaxTiles; ++j) {
          if (j >= nt) break;
          uint8_t *pt = pb + j * GE::kPBytes;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float msub = m_cur[h] == kNegInf ? 0.f : m_cur[h];
            const float pv = fast_exp2(t[j][h] - msub);
            if constexpr (kSplit) {
              // hi = p truncated to bf16, lo = (p - hi) truncated; hi + lo is within 2^-15 of p
              const uint32_t hi = __float_as_uint(pv) & 0xffff0000u;
              const float lo = pv - __uint_as_float(hi);
              *reinterpret_cast<uint16_t *>(pt + h * 128 + ((ck ^ (h & 7)) << 4)) = (uint16_t)(hi >> 16);
              *reinterpret_cast<uint16_t *>(pt + (G + h) * 128 + ((ck ^ ((G + h) & 7)) << 4)) =
                  (uint16_t)(__float_as_uint(lo) >> 16);
              l_part[h] += pv;
            } else {   // f16 operands
              const __half hv = __float2half_rn(pv);
              *reinterpret_cast<__half *>(pt + h * 128 + ((ck ^ (h & 7)) << 4)) = hv;
              l_part[h] += __half2float(hv);
            }
          }
        }
        fence_async_smem();
        mbar_arrive(&p_full[b]);
      }
      // epilogue of the previous unit
      if (prev.valid) {
        const int bp = (u - 1) & 1;
        ok = wait_all(&o_full[bp], ((u - 1) >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        float o[kNO];
        if (num_tiles(prev) > 0) {
          tmem_ld_cols<kNO>(col_o(bp) + lane_base, o);
        } else {
#pragma unroll
          for (int i = 0; i < kNO; ++i) o[i] = 0.f;
        }
        tc_fence_before();
        mbar_arrive(&o_free[bp]);
        const int64_t head0 = (int64_t)prev.row * hq + (int64_t)prev.kvh * gr;
        const int d = tid;            // with head_dim 64, lanes 64..127 repeat 0..63: not stored
        // the two column halves of O^T: bf16 p = hi + lo; fp8 256 p = hi + lo / 16
        auto o_val = [&](int h) {
          return kSplit ? o[h] + o[G + h] : kFp8 ? fmaf(o[G + h], 0.0625f, o[h]) * (1.f / 256.f) : o[h];
        };
        if (prev.nparts == 1) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float val = o_val(h);
            const float om = p.v_hs ? p.out_mult * __ldg(p.v_hs + prev.kvh) : p.out_mult;
            const float inv = l_prev[h] > 0.f ? om / l_prev[h] : 0.f;
            if (d < kD && h < gr) store_out<QT>(p.out, (head0 + h) * kD + d, p.out_f32 != 0, val * inv);
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (d < kD && h < gr) p.ws_acc[((head0 + h) * p.max_partitions + prev.part) * kD + d] = o_val(h);
          if (tid < gr) {
            float mv = m_prev[0], lv = l_prev[0];
#pragma unroll
            for (int h = 1; h < G; ++h)
              if (tid == h) {
                mv = m_prev[h];
                lv = l_prev[h];
              }
            p.ws_ml[(head0 + tid) * p.max_partitions + prev.part] = make_float2(mv, lv);
          }
        }
        if (prev.nparts > 1 && !hand_over(prev.row, prev.kvh, prev.nparts)) {
          ok = false;
          break;
        }
        if (tid == 0) mbar_arrive(&info_free[(u - 1) % kInfo]);
      }
      if (!cur.valid) break;
      prev = cur;
#pragma unroll
      for (int h = 0; h < G; ++h) m_prev[h] = m_cur[h];
    }
    if (ok) {
      hand_over(0, 0, -1);
      drain();
    }
  } else if (warp == kLoadWarp || (warp >= kLoadWarp1 && warp < kLoadWarp1 + NL - 1)) {
    // ===================================================== loaders (two warps)
    // Q^T with cp.async (16-bit caches); every K and V tile with one
    // bulk-tensor box per cache block holding keys of the unit (tiles start on
    // block boundaries), straight into a ring slot in the MMA's layout: 16-bit
    // caches bs / 8 atoms per box, fp8 bs rows of 128 codes per box.  The K
    // warp and the V warp walk the same units and ring positions, each
    // filling its own tiles' slots.
    const int bs = p.block_size;
    const int ldr = warp == kLoadWarp ? 0 : warp - kLoadWarp1 + 1;   // this warp's share: positions = ldr mod NL
    bool ok = true;
    auto issue_tile = [&](const UnitHdr &un, int info_idx, int j, bool is_k, int slot) {
      uint64_t *full_bar = &slot_full[slot];
      const int nvalid = min(kKeys, un.ntok - j * kKeys);
      bool issue = false;
      int32_t bi = 0;
      if (lane < (nvalid + bs - 1) / bs) {
        bi = reinterpret_cast<const volatile int32_t *>(info[info_idx].blk)[8 * j + lane * (bs >> 4)];
        issue = bi >= 0;   // an out-of-range id was reported by the scheduler; its keys stay unread
      }
      const uint32_t boxes = __popc(__ballot_sync(0xffffffffu, issue));
      const CUtensorMap *map = is_k ? tmap_k : tmap_v;
      if constexpr (!kFp8) {
        const int atoms = bs >> 3;
        if (lane == 0) mbar_arrive_expect_tx(full_bar, boxes * atoms * kAtomB);
        __syncwarp();
        if (issue) {
          uint8_t *dst = smem + GE::kOffRing + slot * GE::kSlotBytes + lane * atoms * kAtomB;
          if constexpr (kD == 128) tma_load_4d(dst, map, full_bar, 0, 0, 0, (bi * hkv + un.kvh) * atoms);
          else tma_load_3d(dst, map, full_bar, 0, 0, (bi * hkv + un.kvh) * atoms);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(full_bar, boxes * bs * kD);
        __syncwarp();
        if (issue)
          tma_load_2d(smem + GE::kOffRing + slot * GE::kSlotBytes + lane * bs * kD, map, full_bar, 0,
                      (bi * hkv + un.kvh) * bs);
      }
    };
    // Q^T rows of a unit (16-bit caches): the G query heads of the KV head, 2 * kD bytes each
    auto load_q = [&](const UnitHdr &cur, int b) {
#pragma unroll
      for (int e = lane; e < G * kRowChunks; e += 32) {
        const int h = e / kRowChunks, c16 = e % kRowChunks;
        const bool real = !kPadRows || h < gr;   // padding rows are zero-filled (nothing read)
        const char *src = static_cast<const char *>(p.q) +
                          (real ? (((int64_t)cur.row * hq + (int64_t)cur.kvh * gr + h) * kD) * 2 + c16 * 16 : 0);
        cp_async16(smem + GE::kOffQ + b * GE::kQBytes + (c16 >> 3) * (kNS * 128) + h * 128 +
                       (((c16 & 7) ^ (h & 7)) << 4),
                   src, real ? 16u : 0u);
      }
      cp_async_arrive_noinc(&q_full[b]);
    };
    // one ring, tiles in the MMAs' order: K tiles of unit u, then V tiles of unit u-1
    uint32_t g_pos = 0;   // ring position of the unit's first K tile
    UnitHdr prev;
    prev.valid = 0;
    for (int u = 0; ok; ++u) {
      const int ib = u % kInfo, ibp = (u + kInfo - 1) % kInfo, b = u & 1;
      ok = wait_all(&info_full[ib], (u / kInfo) & 1);
      if (!ok) break;
      const UnitHdr cur = read_unit(&info[ib]);
      const int ntc = num_tiles(cur), ntp = num_tiles(prev);
      if (ldr == 0 && !kFp8 && cur.valid) {
        if (u >= 2) {
          ok = wait_all(&q_free[b], ((u >> 1) - 1) & 1);
          if (!ok) break;
        }
        load_q(cur, b);
      }
      for (int i = (int)((uint32_t)(ldr + NL) - g_pos % NL) % NL; i < ntc + ntp && ok; i += NL) {
        const bool is_k = i < ntc;
        const uint32_t g = g_pos + (uint32_t)i;
        const int slot = (int)(g % S);
        if (g >= (uint32_t)S) ok = wait_all(&slot_free[slot], ((g / S) - 1) & 1);
        if (!ok) break;
        issue_tile(is_k ? cur : prev, is_k ? ib : ibp, is_k ? i : i - ntc, is_k, slot);
      }
      if (!ok) break;
      // this loader is done with unit u-1's descriptor (its V tiles' block ids): a loader
      // may own no tile of several units in a row, and the descriptor must not be
      // reused before it has passed them
      __syncwarp();
      if (u >= 1 && lane == 0) mbar_arrive(&info_free[ibp]);
      g_pos += (uint32_t)(ntc + ntp);
      if (!cur.valid) break;
      prev = cur;
    }
    cp_async_wait_all();
    if (ok) drain();
  } else if (warp == kSchedWarp) {
    // ===================================================== scheduler
    // kClaim units per claim (one atomic step), published in order: two with an
    // fp8 cache, whose units are short, one with a 16-bit cache (measured: 70B
    // bf16 0.272 -> 0.269 ms with one, fp8 0.216 -> 0.220 ms); the block
    // id of run (lane & 7) of tile (lane >> 3) is read by lane `lane`.  fp8:
    // the unit's query scale from the largest |q| of its G query rows.
    const int bs = p.block_size;
    const int total_units = __ldcg(&p.hdr->num_items) * hkv;
    const int64_t cap = min((int64_t)p.max_blocks_per_seq * bs, (int64_t)p.max_partitions * p.partition_size);
    bool ok = true;
    // Store a new token's 16 bytes x (lanes 0-15: K, 16-31: V; elements 8c ..
    // 8c+7; fp8: e4m3(fp32(x) / sc) with an IEEE division, as the cache-write
    // kernel) at cache row crow = (block * Hkv + kvh) * bs + offset, then order
    // the generic stores before the bulk copies that read them (issued by the
    // loader after it acquires the unit's descriptor).
    auto store_new = [&](uint4 x, float sc, int64_t crow) {
      const int side = lane >> 4, c = lane & 15;
      if constexpr (!kFp8) {
        if (c < kD / 8)   // head_dim 64: 8 chunks per row
          *reinterpret_cast<uint4 *>(static_cast<QT *>(const_cast<void *>(side ? tp.v_cache : tp.k_cache)) +
                                     crow * kD + c * 8) = x;
      } else if (c < kD / 8) {   // head_dim 64: 8 chunks per row
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = unpack2(w[k], QT{});
          const uint32_t pair =
              __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(f.x, sc), __fdiv_rn(f.y, sc)), __NV_SATFINITE, __NV_E4M3);
          if (k & 1) o[k >> 1] |= pair << 16;
          else o[k >> 1] = pair;
        }
        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(const_cast<void *>(side ? tp.v_cache : tp.k_cache)) +
                                   crow * kD + c * 8) = make_uint2(o[0], o[1]);
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");   // generic stores -> the async proxy's copies
    };
    constexpr int kClaim = kFp8 ? 2 : 1;
    static_assert(kClaim <= kClaimMax && kInfo % kClaim == 0, "claims of 1 or 2 units");
    for (int u = 0; ok; u += kClaim) {
      for (int k = 0; k < kClaim && ok; ++k)
        if (u + k >= kInfo) ok = wait_all(&info_free[(u + k) % kInfo], (((u + k) / kInfo) - 1) & 1);
      if (!ok) break;
      int id0 = 0;
      if (lane == 0) id0 = atomicAdd(&p.hdr->next_unit, kClaim);
      id0 = __shfl_sync(0xffffffffu, id0, 0);
      // lane k < kClaim resolves unit id0 + k
      const int id = id0 + (lane & (kClaim - 1));
      const bool valid = lane < kClaim && id < total_units;
      int item = 0, L = 0;
      if (valid) item = __ldg(p.items + id / hkv);
      const int row = item >> 12, part = item & 4095;
      if (valid) {
        L = __ldg(p.seq_lens + row);
        if (L < 0 || L > cap) L = L < 0 ? 0 : (int)cap;   // reported by the plan kernel
      }
      const int tok_begin = part * p.partition_size;
      const int ntok = valid ? max(0, min(L, tok_begin + p.partition_size) - tok_begin) : 0;
      const int nparts = max(1, (L + p.partition_size - 1) / p.partition_size);
      bool any_invalid = false;
#pragma unroll
      for (int k = 0; k < kClaim; ++k) {
        const int vk = __shfl_sync(0xffffffffu, (int)valid, k);
        const int rk = __shfl_sync(0xffffffffu, row, k);
        const int tb = __shfl_sync(0xffffffffu, tok_begin, k);
        const int nk = __shfl_sync(0xffffffffu, ntok, k);
        const int kvk = __shfl_sync(0xffffffffu, id % hkv, k);
        const int pk = __shfl_sync(0xffffffffu, part, k);
        const int npk = __shfl_sync(0xffffffffu, nparts, k);
        // fused step: the row's new token goes with its last partition; its loads
        // are in flight with the block-table reads below
        const bool wr = tp.k_new != nullptr && vk && pk == npk - 1;
        int64_t new_slot = -1;
        uint4 new_x = make_uint4(0, 0, 0, 0);
        float new_sc = 1.f;
        if (wr) {
          const int side = lane >> 4;
          new_slot = __ldg(tp.new_slots + rk);
          if ((lane & 15) < kD / 8)
            new_x = __ldg(reinterpret_cast<const uint4 *>(static_cast<const QT *>(side ? tp.v_new : tp.k_new) +
                                                          (int64_t)rk * tp.new_stride + (int64_t)kvk * kD +
                                                          (lane & 15) * 8));
          if (kFp8) new_sc = p.k_hs ? __ldg((side ? p.v_hs : p.k_hs) + kvk) : side ? tp.v_scale : tp.k_scale;
        }
        int32_t qscale = 0;
        if constexpr (kFp8) {
          // Q^T of the unit, in the buffer of its descriptor (free: the descriptor's
          // last reader released it): q 2^e = hi + lo / 16; elements d .. d+7 of
          // head h are bytes d .. d+7 of rows h and G + h (rows of kD bytes,
          // 16-byte chunk c of row r at chunk c ^ (r & 7) with kD 128, or
          // c ^ ((r >> 1) & 3) with kD 64: the 128- and 64-byte swizzles)
          constexpr int kQIt = G * kD / 256;   // 16-byte query chunks per lane
          constexpr int kCPH = kD / 8;         // chunks per head
          auto qoff = [](int r, int c16) {
            return kD == 128 ? r * 128 + (((c16 >> 1) ^ (r & 7)) << 4) : r * 64 + (((c16 >> 1) ^ ((r >> 1) & 3)) << 4);
          };
          uint4 qw[kQIt];
          float amax = 0.f;
          const char *q0 = static_cast<const char *>(p.q) + ((int64_t)rk * hq + (int64_t)kvk * gr) * kD * 2;
#pragma unroll
          for (int i = 0; i < kQIt; ++i) {
            const bool real = !kPadRows || (lane + 32 * i) / kCPH < gr;   // padding rows: zeros
            qw[i] = vk && real ? ld_nc16(q0 + (lane + 32 * i) * 16) : make_uint4(0, 0, 0, 0);
            amax = fmaxf(amax, absmax8(qw[i], QT{}));
          }
#pragma unroll
          for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
          qscale = query_scale_bits(amax);
          if (vk) {
            const float qs = __int_as_float(qscale);
            uint8_t *qb = smem + GE::kOffQ + ((u + k) % kInfo) * GE::kQBytes;
#pragma unroll
            for (int i = 0; i < kQIt; ++i) {
              const int e = lane + 32 * i, h = e / kCPH, c16 = e % kCPH, lr = G + h, half = (c16 & 1) * 8;
              const uint32_t ws[4] = {qw[i].x, qw[i].y, qw[i].z, qw[i].w};
              uint32_t hi[4], lo[4], lo2[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const float2 f = unpack2(ws[c], QT{});
                if constexpr (kQTerms == 3) split3_e4m3(make_float2(f.x * qs, f.y * qs), hi[c], lo[c], lo2[c]);
                else split2_e4m3(make_float2(f.x * qs, f.y * qs), hi[c], lo[c]);
              }
              *reinterpret_cast<uint2 *>(qb + qoff(h, c16) + half) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
              *reinterpret_cast<uint2 *>(qb + qoff(lr, c16) + half) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
              if constexpr (kQTerms == 3) {
                const int r3 = 2 * G + h;
                *reinterpret_cast<uint2 *>(qb + qoff(r3, c16) + half) =
                    make_uint2(lo2[0] | (lo2[1] << 16), lo2[2] | (lo2[3] << 16));
              }
            }
            fence_async_smem();   // generic stores -> the MMAs' reads (after the descriptor's release)
          }
        }
        TcUnit *dst = &info[(u + k) % kInfo];
        const int key0 = tb + (lane >> 3) * kKeys + 16 * (lane & 7);
        int32_t blk = -1;
        if (vk && key0 < tb + nk) {
          const int32_t bi = __ldg(p.block_tables + (int64_t)rk * p.max_blocks_per_seq + key0 / bs);
          if (bi < 0 || bi >= p.num_blocks) record_error(p.err, PA_ERR_DEVICE_CHECK);
          else blk = bi;
        }
        dst->blk[lane] = blk;
        // fused step: the row's new token, for this KV head, stored before the
        // unit that reads it (the row's last partition) is published
        if (wr && new_slot >= 0) {
          const int pos = tb + nk - 1;
          const int32_t bi = __shfl_sync(0xffffffffu, blk, max(nk - 1, 0) >> 4);
          if (nk == 0 || bi < 0 || new_slot != (int64_t)bi * bs + pos % bs) {
            // an empty row has no last position to hold the token; else the slot must be its
            if (lane == 0) record_error(p.err, PA_ERR_DEVICE_CHECK);
          } else {
            store_new(new_x, new_sc, ((int64_t)bi * hkv + kvk) * bs + pos % bs);
          }
        }
        if (lane == k) {
          dst->valid = vk;
          dst->row = rk;
          dst->kvh = vk ? kvk : 0;
          dst->part = part;
          dst->tok_begin = tb;
          dst->ntok = nk;
          dst->nparts = nparts;
          dst->qscale = qscale;
        }
        any_invalid |= !vk;
      }
      __syncwarp();
      for (int k = 0; k < kClaim; ++k) mbar_arrive(&info_full[(u + k) % kInfo]);
      if (any_invalid) break;   // the ids only grow: every later claim is past the end too
    }
    if (ok) drain();
  } else if (warp == kMergeWarp) {
    // ===================================================== merge (last warp)
    // Two duties, polled in turn so that neither waits on the other:
    //  * the CTA's split units (reports from its softmax warps, in order): one
    //    release count per unit on its row's counter publishes the partials; the
    //    count that completes a row acquires every partition's results (fence)
    //    and appends the row to the grid-wide merge list (record, then a release
    //    flag);
    //  * records of the merge list, claimed in the order they were appended and
    //    merged (merge_job), so every CTA's merge warp shares the merging.
    // Waiting without progress on either is bounded (PA_ERR_TIMEOUT).
    // With kSepMerge another warp merges from the start, and this one only
    // counts: a merge (one or more dependent L2 round trips, several µs under
    // the decode's memory load) no longer delays the appends behind it.
    const int total_jobs = __ldcg(&p.hdr->pad[2]);
    int nrep = 0, t = -1;
    bool local_done = false, list_done = kSepMerge;
    uint64_t t_idle = global_timer_ns();
    for (;;) {
      if (*abort_flag) break;
      if (local_done && list_done && t < 0) break;
      bool progress = false;
      if (!local_done) {
        const int rs = nrep % kRep;
        int got = 0;
        if (lane == 0) got = mbar_try_wait(&rep_full[rs], (nrep / kRep) & 1) ? 1 : 0;
        if (__shfl_sync(0xffffffffu, got, 0)) {
          if (lane == 0) {
            const int4 r = reports[rs];
            if (r.z < 0) {
              got = 2;
            } else {
              int old;
              asm volatile("atom.release.gpu.global.add.s32 %0, [%1], 1;"
                           : "=r"(old)
                           : "l"(p.ws_count + (int64_t)r.x * hq + (int64_t)r.y * gr)
                           : "memory");
              if (old == r.z - 1) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                const int jt = atomicAdd(&p.hdr->pad[0], 1);
                asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(&tp.jobs[jt].word), "l"(merge_word(r.x, r.y, r.z))
                             : "memory");
              }
              mbar_arrive(&rep_free[rs]);
            }
          }
          if (__shfl_sync(0xffffffffu, got, 0) == 2) local_done = true;
          ++nrep;
          progress = true;
        }
      }
      if (t < 0 && !list_done) {
        if (lane == 0) t = atomicAdd(&p.hdr->pad[1], 1);
        t = __shfl_sync(0xffffffffu, t, 0);
        if (t >= total_jobs) {
          list_done = true;
          t = -1;
        }
      }
      uint64_t word = 0;
      if (t >= 0 && lane == 0)
        asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(word) : "l"(&tp.jobs[t].word) : "memory");
      if (!__shfl_sync(0xffffffffu, word != 0, 0)) {
        if (progress) {
          t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
          if (lane == 0) record_error(p.err, PA_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        } else {
          __nanosleep(500);
        }
        continue;
      }
      merge_job(word);
      t = -1;
      t_idle = global_timer_ns();
    }
    if constexpr (kSepMerge) drain();
  } else if (kSepMerge && warp == kMerge2Warp) {
    // ===================================================== merging (kSepMerge)
    drain();
  } else if (warp == kMmaWarp) {
    // ===================================================== MMA issue
    // The whole warp runs the schedule (descriptors stay warp-uniform); one
    // elected lane issues the MMAs and their commits.
    const bool leader = elect_one();
    const uint32_t idesc_s = umma_idesc(kAB, kNS, false, false);
    const uint32_t idesc_o = umma_idesc(kAB, kNO, false, true);
    // one MMA: kind::f8f6f4 for an fp8 cache, else kind::f16
    auto mma = [&](uint32_t d, uint64_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
      if constexpr (kFp8) umma_f8(d, a, bdesc, idesc, acc);
      else umma(d, a, bdesc, idesc, acc);
    };
    const uint32_t ring = smem_u32(smem + GE::kOffRing);
    const uint32_t qbuf = smem_u32(smem + GE::kOffQ);
    const uint32_t pbuf = smem_u32(smem + GE::kOffP);
    // Operand descriptors: built once; a tile, buffer or k step adds its byte
    // offset / 16 to the start-address field (every address stays below 256 KB,
    // so the 14-bit field never carries).  One thread issues every MMA, and each
    // instruction on its path delays the next issue.
    auto dofs = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
    // fp8 with head_dim 64: K, V and Q^T in 64-byte rows (64-byte swizzle, 8-row groups 512 B
    // apart); V^T's second 64-element half of M repeats the first (LBO 0), as with 16-bit V
    constexpr bool kSw64 = kFp8 && kD == 64;
    const uint64_t kdesc0 = kSw64 ? umma_desc_sw64(ring, 16, 512) : kFp8 ? umma_desc(ring, 16) : umma_desc_sbo(ring, 16, kAtomB);
    const uint64_t vdesc0 = kSw64  ? umma_desc_sw64(ring, 0, 512)
                            : kFp8 ? umma_desc_sbo(ring, 1024, 1024)
                                   : umma_desc_sbo(ring, kD == 128 ? 1024 : 0, kAtomB);
    const uint64_t qdesc0 = kSw64 ? umma_desc_sw64(qbuf, 16, 512) : umma_desc(qbuf, 16), pdesc0 = umma_desc(pbuf, 16);
    uint32_t g_cons = 0;   // tiles consumed, in the ring's order
    bool ok = true, issued = false;
    UnitHdr prev;
    prev.valid = 0;
    for (int u = 0; ok; ++u) {
      const int ib = u % kInfo, b = u & 1;
      ok = wait_all(&info_full[ib], (u / kInfo) & 1);
      if (!ok) break;
      const UnitHdr cur = read_unit(&info[ib]);
      if (cur.valid) {
        // S^T(u, j) = K_j . Q^T into buffer b (its previous reader: the softmax of u-2)
        const int nt = num_tiles(cur);
        if (u >= 2) {
          ok = wait_all(&s_free[b], ((u >> 1) - 1) & 1);
          if (!ok) break;
        }
        if constexpr (!kFp8) {   // fp8: Q^T was written (and fenced) with the descriptor
          ok = wait_all(&q_full[b], (u >> 1) & 1);
          if (!ok) break;
          fence_async_smem();   // Q^T staged by cp.async (generic proxy) -> the MMAs' reads
        }
        for (int j = 0; j < nt; ++j) {
          const int slot = (int)(g_cons % S);
          ok = wait_all(&slot_full[slot], (g_cons / S) & 1);
          if (!ok) break;
          tc_fence_after();   // the tile came by bulk copy (async proxy): no proxy fence
          if (leader) {
            const uint64_t kd = kdesc0 + dofs(slot * GE::kSlotBytes), qd = qdesc0 + dofs((kFp8 ? ib : b) * GE::kQBytes);
            const uint32_t dcol = col_s(b, j);
            if constexpr (kFp8) {
              // 32 elements (32 B of each kD-byte row) per MMA
#pragma unroll
              for (int k = 0; k < kD / 32; ++k) mma(dcol, kd + dofs(k * 32), qd + dofs(k * 32), idesc_s, k > 0 ? 1u : 0u);
            } else {
#pragma unroll
              for (int k = 0; k < kD / 16; ++k)
                mma(dcol, kd + dofs((k >> 2) * 1024 + (k & 3) * 32), qd + dofs((k >> 2) * (kNS * 128) + (k & 3) * 32),
                    idesc_s, k > 0 ? 1u : 0u);
            }
            umma_commit(&slot_free[slot]);
          }
          __syncwarp();
          issued = true;
          ++g_cons;
        }
        if (!ok) break;
        if (leader) {
          umma_commit(&s_full[b]);
          if constexpr (!kFp8) umma_commit(&q_free[b]);
        }
        __syncwarp();
      }
      if (prev.valid) {
        // O^T(u-1) = sum_j V_j^T . P_j^T (its previous reader: the epilogue of u-3)
        const int bp = (u - 1) & 1, nt = num_tiles(prev);
        ok = wait_all(&p_full[bp], ((u - 1) >> 1) & 1);
        if (!ok) break;
        if (u - 1 >= 2) {
          ok = wait_all(&o_free[bp], (((u - 1) >> 1) - 1) & 1);
          if (!ok) break;
        }
        for (int j = 0; j < nt; ++j) {
          const int slot = (int)(g_cons % S);
          ok = wait_all(&slot_full[slot], (g_cons / S) & 1);
          if (!ok) break;
          // keys past the end of the unit take part only up to the end of their
          // key group (16 keys per MMA, 32 with fp8); their rows in that group may
          // hold stale values (a whole atom or cache block is copied, and copies
          // of later ones are skipped), so they are zeroed: P is 0 there, and
          // 0 * NaN would not be
          constexpr int kGroup = kFp8 ? 32 : 16;
          const int nvalid = min(kKeys, prev.ntok - j * kKeys);
          const int ngroups = (nvalid + kGroup - 1) / kGroup;
          uint8_t *vt = smem + GE::kOffRing + slot * GE::kSlotBytes;
          if (nvalid % kGroup) {
            if constexpr (kFp8) {
              constexpr int kRowC = kD / 16;   // 16-byte chunks of a kD-byte row
              for (int e = lane; e < (kGroup * ngroups - nvalid) * kRowC; e += 32)
                *reinterpret_cast<uint4 *>(vt + (nvalid + e / kRowC) * kD + (e % kRowC) * 16) = make_uint4(0, 0, 0, 0);
            } else {
              for (int e = lane; e < (kGroup * ngroups - nvalid) * kRowChunks; e += 32) {
                const int r = nvalid + e / kRowChunks, c = e % kRowChunks;   // row, 16-byte chunk of it
                *reinterpret_cast<uint4 *>(vt + (r >> 3) * kAtomB + (c >> 3) * 1024 + (r & 7) * 128 +
                                           (c & 7) * 16) = make_uint4(0, 0, 0, 0);
              }
            }
            fence_async_smem();   // the zeroed rows (generic proxy) -> the MMAs' reads
            __syncwarp();
          }
          // P^T was fenced by the softmax warps before p_full; the tile came by bulk copy
          tc_fence_after();
          if (leader) {
            const uint64_t vd = vdesc0 + dofs(slot * GE::kSlotBytes), pd = pdesc0 + dofs((bp * kMaxTiles + j) * GE::kPBytes);
            const uint32_t dcol = col_o(bp), acc0 = j > 0 ? 1u : 0u;
            // unrolled over a whole tile's key groups, the tail's predicated off
            if constexpr (kFp8) {
              // V^T: one kD-element MN panel, 8-key groups 8 kD bytes apart, 32 keys per MMA
#pragma unroll
              for (int kk = 0; kk < kKeys / 32; ++kk)
                if (kk < ngroups) mma(dcol, vd + dofs(kk * 32 * kD), pd + dofs(kk * 32), idesc_o, kk > 0 ? 1u : acc0);
            } else {
              // M = 128 elements of V^T in two 64-element halves (LBO apart): panels 0 and 1,
              // or panel 0 twice with head_dim 64 (lanes 64..127 of O^T then repeat 0..63)
#pragma unroll
              for (int kk = 0; kk < kKeys / 16; ++kk)
                if (kk < ngroups)
                  mma(dcol, vd + dofs(kk * 2 * kAtomB), pd + dofs((kk >> 2) * (kNO * 128) + (kk & 3) * 32), idesc_o,
                      kk > 0 ? 1u : acc0);
            }
            umma_commit(&slot_free[slot]);
          }
          __syncwarp();
          issued = true;
          ++g_cons;
        }
        if (!ok) break;
        if (leader) {
          umma_commit(&o_full[bp]);
          mbar_arrive(&info_free[(u - 1) % kInfo]);
        }
        __syncwarp();
      }
      if (!cur.valid) break;
      prev = cur;
    }
    // every MMA issued above is complete before tensor memory is freed
    if (issued) {
      if (leader) umma_commit(fin);
      __syncwarp();
      mbar_wait(fin, 0, p.err);
    }
    if (ok) drain();
  }

  // ===================================================== teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(GE::kTmemCols));
  }
}

template <typename KV, typename QT, int G, int D, bool kPadRows>
__global__ void __launch_bounds__(dtc::Roles::threads_for(dtc::Roles::loaders(G), dtc::Roles::sep_merge(G)), 1)
    decode_tc_kernel(const DecodeTcParams tp, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v) {
  decode_tc_body<KV, QT, G, D, dtc::Roles::loaders(G), dtc::Roles::sep_merge(G), kPadRows>(tp, &tmap_k, &tmap_v);
}

// One CTA: count the split rows' merges and clear the merge list, and list
// the (row, partition) items -- rows with the most partitions
// first, then the single-partition rows by their number of 128-key tiles
// (a counting sort; rows of equal key in any order), each row's partitions
// together and in order -- and reset the scheduling cursor and the split
// rows' completion counters.  Long rows are then finished, and merged, while
// shorter ones still run, and the smallest units come last, which evens out
// the CTAs' finishing times.  An empty row lists one item of zero tokens.
template <int kUnused>
__global__ void __launch_bounds__(1024) decode_tc_plan_kernel(DecodeParams p, DecodeMergeJob *jobs) {
  // launched as a programmatic dependent of what precedes it on the stream
  // (the previous step's decode among others): its launch overlaps that grid's
  // end, and nothing of the workspace is touched before that grid is complete
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the decode grid may launch now: it sets itself up, then waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // sort key 0 .. maxp + 3: 3 + nparts for a split row, else its tiles (0 .. 4);
  // base[maxp + 3 - key]: items of the key (descending), then its next free item
  __shared__ int base[kMaxPartitions + 4];
  const int tid = threadIdx.x;
  const int maxp = p.max_partitions;
  const int nkeys = maxp + 4;
  __shared__ int split_rows;
  for (int64_t i = tid; i < (int64_t)p.num_seqs * p.num_q_heads; i += blockDim.x) p.ws_count[i] = 0;
  if (p.max_partitions > 1)   // the merge list exists only when a row can be split
    for (int64_t i = tid; i < (int64_t)p.num_seqs * p.num_kv_heads; i += blockDim.x) jobs[i].word = 0;
  for (int i = tid; i < nkeys; i += blockDim.x) base[i] = 0;
  if (tid == 0) split_rows = 0;
  __syncthreads();
  auto len_of = [&](int r, bool report) { return checked_len(p, r, report); };
  auto nparts_of = [&](int L) { return max(1, (L + p.partition_size - 1) / p.partition_size); };
  auto slot_of = [&](int L, int np) { return nkeys - 1 - (np > 1 ? 3 + np : (L + dtc::kKeys - 1) / dtc::kKeys); };
  for (int r = tid; r < p.num_seqs; r += blockDim.x) {
    const int L = len_of(r, true), np = nparts_of(L);
    atomicAdd(&base[slot_of(L, np)], np);
    if (np > 1) atomicAdd(&split_rows, 1);
  }
  __syncthreads();
  if (tid == 0) {   // exclusive scan (a small serial pass)
    int run = 0;
    for (int i = 0; i < nkeys; ++i) {
      const int c = base[i];
      base[i] = run;
      run += c;
    }
    p.hdr->num_items = run;
    p.hdr->next_unit = 0;
    p.hdr->pad[0] = 0;                              // merge records appended
    p.hdr->pad[1] = 0;                              // merge records taken
    p.hdr->pad[2] = split_rows * p.num_kv_heads;    // one per split (row, KV head)
  }
  __syncthreads();
  for (int r = tid; r < p.num_seqs; r += blockDim.x) {
    const int L = len_of(r, false), np = nparts_of(L);
    const int at = atomicAdd(&base[slot_of(L, np)], np);
    for (int q = 0; q < np; ++q) p.items[at + q] = (r << 12) | q;
  }
}

// Host launcher: the plan kernel, then one persistent CTA per SM launched as its
// programmatic dependent.
// The plan kernel, launched as a programmatic dependent of the stream's
// previous work (it waits for that work before touching anything).
template <int kUnused = 0>
cudaError_t launch_decode_tc_plan(const DecodeParams &d, DecodeMergeJob *jobs, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_plan_kernel<0>, d, jobs);
}

template <typename KV, typename QT, int G, int D, bool kPadRows>
cudaError_t launch_decode_tc_one(const DecodeTcParams &p, const PoolMaps &m, cudaStream_t s) {
  constexpr bool kSplit = std::is_same<QT, __nv_bfloat16>::value && !std::is_same<KV, uint8_t>::value;
  constexpr int smem =
      dtc::TcGeo<G, kSplit, std::is_same<KV, uint8_t>::value, dtc::QTerms<KV, QT>::value, D>::kSmemBytes;
  cudaError_t e = launch_decode_tc_plan(p.d, p.jobs, s);
  if (e != cudaSuccess) return e;
  if ((e = ensure_smem_limit<decode_tc_kernel<KV, QT, G, D, kPadRows>>(smem)) != cudaSuccess) return e;
  int sms = 0;
  if ((e = current_sm_count(&sms)) != cudaSuccess) return e;
  // programmatic dependent launch: the decode grid's set-up overlaps the plan kernel
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(dtc::Roles::threads_for(dtc::Roles::loaders(G), dtc::Roles::sep_merge(G)));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<KV, QT, G, D, kPadRows>, p, m.k, m.v);
}

// m: tensor maps over the pools, one box per cache block of one KV head: 16-bit
// caches viewed as [atoms of 8 rows][2 panels][8 rows][64] (head_dim 128) or
// [atoms of 8 rows][8 rows][64] (head_dim 64), fp8 caches as [rows][128]
// (128-byte swizzle).
// kPadRows false: gqa is exactly 4, 8 or 16 (head_dim 64: 4 or 8), every head index compile-time;
// true: any other group of 1..16 (1..8), run in the kernel for the next of those sizes.
template <typename KV, typename QT, bool kPadRows>
cudaError_t launch_decode_tc(const DecodeTcParams &p, int gqa, int head_dim, const PoolMaps &m, cudaStream_t s) {
  // a group of gqa query heads runs in the kernel for the next of 4, 8 or 16 rows
  if (gqa < 1) return cudaErrorInvalidValue;
  if (decode_tc_exact_group(head_dim, gqa) == kPadRows) return cudaErrorInvalidValue;
  if (head_dim == 64) {
    if (gqa <= 4) return launch_decode_tc_one<KV, QT, 4, 64, kPadRows>(p, m, s);
    if (gqa <= 8) return launch_decode_tc_one<KV, QT, 8, 64, kPadRows>(p, m, s);
    return cudaErrorInvalidValue;
  }
  if (head_dim != 128) return cudaErrorInvalidValue;
  if (gqa <= 4) return launch_decode_tc_one<KV, QT, 4, 128, kPadRows>(p, m, s);
  if (gqa <= 8) return launch_decode_tc_one<KV, QT, 8, 128, kPadRows>(p, m, s);
  if (gqa <= 16) return launch_decode_tc_one<KV, QT, 16, 128, kPadRows>(p, m, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa
