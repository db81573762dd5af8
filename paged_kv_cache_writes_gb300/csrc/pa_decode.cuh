// pa_decode.cuh -- paged decode on CUDA cores, persistent and warp-granular.
//
// What it computes: for each sequence (row) and query head h,
//   out[row][h] = sum_p softmax_p(scale * q[row][h] . K[p][g]) V[p][g],
// g = h / (Hq / Hkv), K/V gathered through the block table ("Inside vLLM
// Architecture", sections "Architectural Anatomy: PagedAttention Virtual
// Memory Paging" and "CUDA Shared Memory Optimization in PagedAttention";
// exact attention per its "Semantic FAQ Section").
//
// Work decomposition.  A row of L tokens is cut into partitions of PS tokens
// (split-KV).  A *unit* is (row, partition, KV head, group of HPC query
// heads); the HPC heads share every K/V byte read.  A one-CTA plan kernel
// lists the non-empty (row, partition) items -- full partitions first, then
// the ragged last partitions -- so no work slot is wasted on the tail of a
// short row.  The decode kernel is persistent (one CTA per SM); each of its
// warps is an independent worker that claims units from an atomic cursor.
//
// Inside a warp:
//  * the next unit is claimed while the current one computes: the cursor
//    bump and the two dependent reads behind it (item, then the row's length
//    and block ids) are issued one per tile, so their latency is hidden;
//  * lane 0 keeps a ring of kSlots 16-token K/V tiles in flight with bulk-
//    tensor (TMA) copies, one box per K and per V tile (3D box over both
//    128-byte panels of the 256-byte rows; 128-byte swizzle), running ahead
//    across the boundary into the next claimed unit; the unit's block ids
//    sit one per lane in a register (one coalesced load per unit);
//  * q for the next unit arrives by a 1D bulk copy while the current unit
//    computes, and is widened to fp32, pre-scaled by scale*log2(e);
//  * Q.K^T (HPC >= 4): lane = (quarter of head_dim, token pair), every head
//    of the group; one 16-byte q load from shared memory feeds 2 tokens x 2
//    heads of packed fp32x2 FMAs, and a two-level shuffle reduction over the
//    quarters leaves each lane with its scores (HPC == 1: lane = (half of
//    head_dim, token));
//  * online softmax in the log2 domain with a lazy reference maximum: the
//    accumulators are rescaled only when a tile's maximum exceeds the
//    reference by more than kRescaleLog2 (2^8 headroom in fp32), which
//    leaves the result exact and skips nearly every rescale;
//  * P.V: lane = (token sub-step, 8 output elements), all HPC heads;
//  * a unit of a split row writes (acc, max, sum) to the workspace; the last
//    unit of the row to arrive (atomic counter, reset after use) combines
//    the partitions, sum_p 2^(m_p-M) acc_p / sum_p 2^(m_p-M) l_p.
#pragma once

#include "pa_attention.cuh"

namespace pa {

constexpr float kRescaleLog2 = 8.f;

// Workspace header (first 256 bytes), written by the plan kernel.
struct DecodeHeader {
  int32_t next_unit;   // dynamic scheduling cursor
  int32_t num_items;   // (row, partition) items listed
  int32_t pad[62];
};

template <typename KV, int D, int HPC>
struct DecGeo {
  using G = Geo<KV, D>;
  static constexpr int kStageTok = 16;
  static constexpr int kStageBytes = G::kStageBytes;
  // ~16 KB of tiles per warp: one being computed, the rest in flight.  More
  // warps per SM (9 for bf16 with head_dim 128) beat deeper per-warp rings.
  static constexpr int kSlots = kStageBytes >= 8192 ? 2 : kStageBytes >= 4096 ? 4 : 8;
  static constexpr int kQsOff = kSlots * kStageBytes;               // fp32 [D/2][HPC][2]
  static constexpr int kQrawOff = kQsOff + D * HPC * 4;             // raw q, HPC x D
  static constexpr int kPOff = kQrawOff + HPC * D * 2;              // float2 [16][HPC]
  static constexpr int kBarOff = kPOff + kStageTok * HPC * 8;       // full[kSlots], qbar
  static constexpr int kWarpBytes = (kBarOff + (kSlots + 1) * 8 + 1023) / 1024 * 1024;
  static constexpr int kNW0 = (226 * 1024) / kWarpBytes;
  static constexpr int kNW = kNW0 > 8 ? 8 : kNW0;                   // warps (workers) per CTA
  static constexpr int kSmem = kNW * kWarpBytes + 1024;
  static_assert(kNW >= 1, "per-warp shared memory too large");
};

struct DecodeParams {
  const void *q;
  void *out;
  int32_t out_f32;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  const int32_t *seq_lens;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t groups;            // query-head groups per KV head (G / HPC)
  int32_t block_size;
  int64_t num_blocks;
  int32_t partition_size;    // <= 32 * block_size, multiple of 32
  int32_t max_partitions;
  int32_t tile_shift;        // log2(block_size / 16): 16-token tiles per block
  int32_t kv_rows;           // num_kv_heads * block_size: rows of one block in the 2D pool view
  float q_mult;
  float out_mult;
  const float *k_hs;         // fp8, optional: [Hkv] per-head scales multiplying q_mult / out_mult
  const float *v_hs;
  DecodeHeader *hdr;
  int32_t *items;            // (row << 12) | partition
  float *ws_acc;             // [rows][Hq][max_partitions][D]
  float2 *ws_ml;             // [rows][Hq][max_partitions]
  int32_t *ws_count;         // [rows][Hq]
  int32_t *err;
};

// Clamp a row's length to what its block table and the partition count can
// address, recording the violation.
__device__ __forceinline__ int checked_len(const DecodeParams &p, int row, bool report) {
  int L = __ldg(p.seq_lens + row);
  const int64_t cap = min((int64_t)p.max_blocks_per_seq * p.block_size,
                          (int64_t)p.max_partitions * p.partition_size);
  if (L < 0 || L > cap) {
    if (report) record_error(p.err, PA_ERR_DEVICE_CHECK);
    L = L < 0 ? 0 : (int)cap;
  }
  return L;
}

// One CTA: list (row, partition) items -- every full partition first, then
// each row's ragged last partition (an empty row lists one item of zero
// tokens, whose unit writes a zero output) -- and reset the scheduling
// cursor and the split-KV arrival counters.
template <int kUnused>
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams p) {
  __shared__ int s_full[1024];
  __shared__ int s_part[1024];
  const int tid = threadIdx.x;
  for (int64_t i = tid; i < (int64_t)p.num_seqs * p.num_q_heads; i += blockDim.x) p.ws_count[i] = 0;
  // pass 0: total number of full partitions (the ragged ones are listed after them)
  int tot_full = 0;
  for (int r0 = 0; r0 < p.num_seqs; r0 += 1024) {
    const int r = r0 + tid;
    s_full[tid] = r < p.num_seqs ? checked_len(p, r, true) / p.partition_size : 0;
    __syncthreads();
    for (int off = 512; off > 0; off >>= 1) {
      if (tid < off) s_full[tid] += s_full[tid + off];
      __syncthreads();
    }
    tot_full += s_full[0];
    __syncthreads();
  }
  int base_full = 0, base_part = tot_full;
  for (int r0 = 0; r0 < p.num_seqs; r0 += 1024) {
    const int r = r0 + tid;
    const int L = r < p.num_seqs ? checked_len(p, r, false) : 0;
    const int nfull = r < p.num_seqs ? L / p.partition_size : 0;
    const int npart = r < p.num_seqs && (L % p.partition_size != 0 || L == 0) ? 1 : 0;
    s_full[tid] = nfull;
    s_part[tid] = npart;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // inclusive scans
      const int af = tid >= off ? s_full[tid - off] : 0;
      const int ap = tid >= off ? s_part[tid - off] : 0;
      __syncthreads();
      s_full[tid] += af;
      s_part[tid] += ap;
      __syncthreads();
    }
    const int ex_full = s_full[tid] - nfull, ex_part = s_part[tid] - npart;
    for (int q = 0; q < nfull; ++q) p.items[base_full + ex_full + q] = (r << 12) | q;
    if (npart) p.items[base_part + ex_part] = (r << 12) | nfull;
    const int add_full = s_full[1023], add_part = s_part[1023];
    __syncthreads();
    base_full += add_full;
    base_part += add_part;
  }
  if (tid == 0) {
    p.hdr->num_items = base_part;
    p.hdr->next_unit = 0;
  }
}

// A claimed unit, replicated in every lane (blk: this lane's block id).
struct Unit {
  int valid, row, kvh, h0, part, tok_begin, tok_end, nst, nparts;
  int32_t blk;
};

// A claim in flight.  Its three dependent global reads (cursor -> item ->
// length and block ids) are issued one step at a time between K/V tiles, so
// their latency hides behind the current unit's compute.
struct PendingClaim {
  int phase;  // 0: cursor bumped, 1: item requested, 2: row data requested, 3: resolved
  int id, item, L;
  int32_t blk;
};

__device__ __forceinline__ void claim_start(PendingClaim &c, const DecodeParams &p, int lane) {
  c.id = 0;
  if (lane == 0) c.id = atomicAdd(&p.hdr->next_unit, 1);
  c.phase = 0;
}

// Advance a pending claim by one step (warp-uniform); true once `u` is filled.
template <int HPC>
__device__ __forceinline__ bool claim_step(PendingClaim &c, Unit &u, const DecodeParams &p, int total_units,
                                           int lane) {
  const int hgt = p.num_kv_heads * p.groups;
  if (c.phase == 0) {
    c.id = __shfl_sync(0xffffffffu, c.id, 0);
    if (c.id < total_units) c.item = __ldg(p.items + c.id / hgt);
    c.phase = 1;
    return false;
  }
  if (c.phase == 1) {
    c.blk = -1;
    if (c.id < total_units) {
      const int row = c.item >> 12, part = c.item & 4095;
      c.L = __ldg(p.seq_lens + row);
      const int lb = part * p.partition_size / p.block_size + lane;
      if (lb < p.max_blocks_per_seq) c.blk = __ldg(p.block_tables + (int64_t)row * p.max_blocks_per_seq + lb);
    }
    c.phase = 2;
    return false;
  }
  if (c.phase == 2) {
    u.valid = c.id < total_units;
    u.blk = -1;
    if (u.valid) {
      const int hs = c.id % hgt;
      u.row = c.item >> 12;
      u.part = c.item & 4095;
      u.kvh = hs / p.groups;
      u.h0 = u.kvh * (p.num_q_heads / p.num_kv_heads) + (hs % p.groups) * HPC;
      int L = c.L;
      const int64_t cap = min((int64_t)p.max_blocks_per_seq * p.block_size,
                              (int64_t)p.max_partitions * p.partition_size);
      if (L < 0 || L > cap) L = L < 0 ? 0 : (int)cap;  // reported by the plan kernel
      u.nparts = max(1, (L + p.partition_size - 1) / p.partition_size);
      u.tok_begin = u.part * p.partition_size;
      u.tok_end = min(L, u.tok_begin + p.partition_size);
      u.nst = (u.tok_end - u.tok_begin + 15) >> 4;
      const int nblk = (u.tok_end - u.tok_begin + p.block_size - 1) / p.block_size;
      u.blk = lane < nblk ? c.blk : -1;
    }
    c.phase = 3;
  }
  return true;
}

__device__ __forceinline__ void bulk_load_1d(void *smem_dst, const void *gsrc, uint32_t bytes,
                                             uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Position of q[h][d] (fp32, pre-scaled) in a warp's q buffer.  HPC >= 4:
// d-pair dp = d/2 lies in quarter dq = dp / (D/8) at local index dpl; the 16
// bytes holding heads (2k, 2k+1) of that d-pair for the four quarters are
// adjacent, so the four quarter lanes of a Q.K^T step read one 64-byte run.
// HPC == 1: plain [D] order.
template <int D, int HPC>
__device__ __forceinline__ int q_index(int d, int h) {
  if constexpr (HPC >= 4) {
    const int dp = d >> 1, dq = dp / (D / 8), dpl = dp % (D / 8), k = h >> 1;
    return (((dpl * (HPC / 2) + k) * 4 + dq) * 4) + (h & 1) * 2 + (d & 1);
  } else {
    return d;
  }
}

template <typename KV, typename QT, int D, int HPC>
__global__ void __launch_bounds__(DecGeo<KV, D, HPC>::kNW * 32, 1)
    paged_decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v) {
  using G = Geo<KV, D>;
  using DG = DecGeo<KV, D, HPC>;
  constexpr int S = DG::kSlots;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *wbase = smem + warp * DG::kWarpBytes;
  float *q_s = reinterpret_cast<float *>(wbase + DG::kQsOff);
  QT *q_raw = reinterpret_cast<QT *>(wbase + DG::kQrawOff);
  float2 *p_s = reinterpret_cast<float2 *>(wbase + DG::kPOff);
  uint64_t *full = reinterpret_cast<uint64_t *>(wbase + DG::kBarOff);
  uint64_t *qbar = full + S;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    mbar_init(qbar, 1);
    fence_mbar_init();
    if (warp == 0) {
      prefetch_tensor_map(&tmap_k);
      prefetch_tensor_map(&tmap_v);
    }
  }
  __syncwarp();

  const int total_units = __ldcg(&p.hdr->num_items) * p.num_kv_heads * p.groups;
  const int bs = p.block_size;

  // --------------------------------------------------------------- producer side
  auto issue_q = [&](const Unit &u) {
    if (lane == 0) {  // every lane's reads of q_raw completed before this point
      constexpr uint32_t bytes = HPC * D * sizeof(QT);
      mbar_arrive_expect_tx_relaxed(qbar, bytes);
      bulk_load_1d(q_raw, static_cast<const QT *>(p.q) + ((int64_t)u.row * p.num_q_heads + u.h0) * D,
                   bytes, qbar);
    }
  };
  Unit U0;
  {
    PendingClaim c0;
    claim_start(c0, p, lane);
    while (!claim_step<HPC>(c0, U0, p, total_units, lane)) {
    }
  }
  Unit U1;
  U1.valid = 0;
  U1.blk = -1;
  uint32_t g_issue = 0, g_comp = 0, qphase = 0;

  // Issue target: the unit whose next tile is loaded next (U0, then U1),
  // kept in its own registers with the per-unit address terms precomputed.
  int it_valid = 0, it_nst = 0, it_st = 0, it_row = 0, it_which = 0;
  int32_t it_blk = -1;
  auto set_target = [&](const Unit &u, int which) {
    it_valid = u.valid;
    it_nst = u.valid ? u.nst : 0;
    it_st = 0;
    it_row = u.valid ? u.kvh * bs : 0;
    it_blk = u.blk;
    it_which = which;
  };
  // Tile it_st of the target into slot g_issue % S: one box for K, one for V.
  auto issue_tile = [&]() {
    const int slot = g_issue % S;
    const int32_t blk = __shfl_sync(0xffffffffu, it_blk, it_st >> p.tile_shift);
    if (lane == 0) {  // the slot's previous tile was fully read (its values were consumed)
      if (blk < 0 || blk >= p.num_blocks) {
        record_error(p.err, PA_ERR_DEVICE_CHECK);
        mbar_arrive(&full[slot]);
      } else {
        mbar_arrive_expect_tx_relaxed(&full[slot], G::kStageBytes);
        const int32_t y = blk * p.kv_rows + it_row + ((it_st & ((1 << p.tile_shift) - 1)) << 4);
        uint8_t *st_base = wbase + slot * G::kStageBytes;
        if constexpr (G::kPanels == 2) {  // both 128-byte panels of the rows in one 3D box
          tma_load_3d(st_base, &tmap_k, &full[slot], 0, y, 0);
          tma_load_3d(st_base + G::kTileBytes, &tmap_v, &full[slot], 0, y, 0);
        } else {
          tma_load_2d(st_base, &tmap_k, &full[slot], 0, y);
          tma_load_2d(st_base + G::kTileBytes, &tmap_v, &full[slot], 0, y);
        }
      }
    }
    ++it_st;
    ++g_issue;
  };
  auto fill = [&]() {
    while (g_issue - g_comp < (uint32_t)S && it_valid) {
      if (it_st < it_nst) {
        issue_tile();
      } else if (it_which == 0 && U1.valid) {
        set_target(U1, 1);
      } else {
        break;
      }
    }
  };
  set_target(U0, 0);
  if (U0.valid) issue_q(U0);
  fill();

  bool ok = true;
  while (U0.valid && ok) {
    PendingClaim pc;
    claim_start(pc, p, lane);
    bool have_next = false;
    // q of this unit: widen and pre-scale into q_s (layout: see q_index)
    ok = __all_sync(0xffffffffu, mbar_wait(qbar, qphase, p.err));
    if (!ok) break;
    qphase ^= 1;
    const float qm = p.k_hs ? p.q_mult * __ldg(p.k_hs + U0.kvh) : p.q_mult;
    for (int e8 = lane * 8; e8 < HPC * D; e8 += 256) {
      const uint4 w = *reinterpret_cast<const uint4 *>(q_raw + e8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      const int h = e8 / D, d0 = e8 % D;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2(ws[i], QT{});
        *reinterpret_cast<float2 *>(q_s + q_index<D, HPC>(d0 + 2 * i, h)) = make_float2(f.x * qm, f.y * qm);
      }
    }
    __syncwarp();
    fill();

    // Q.K^T lane mapping (HPC >= 4): lane = dq * 8 + t8 covers tokens t8 and
    // t8 + 8 of the tile, every head of the group, and the dq-th quarter of
    // head_dim.  Each K element is widened once per lane that uses it; each
    // 16-byte q load feeds 2 tokens x 2 heads of FMA pairs, and the 4 quarters
    // read 64 contiguous bytes per wavefront.  A two-level shuffle reduction
    // over dq leaves lane (dq, t8) with token t8 + 8*(dq & 1) and heads
    // (dq >> 1) * HPC/2 + j.  One head (HPC == 1): lane = (d half, token).
    constexpr int HS = HPC >= 4 ? HPC / 2 : 1;  // scores held per lane after the reduction
    const int dq = lane >> 3, t8 = lane & 7;
    const int my_t = HPC >= 4 ? t8 + 8 * (dq & 1) : (lane & 15);
    const int my_h0 = HPC >= 4 ? (dq >> 1) * HS : 0;
    const int hh = lane >> 4;  // HPC == 1: which half of head_dim

    float2 acc[HPC][4];
    float m_ref[HPC];
    float l_part[HS];
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      m_ref[h] = kNegInf;
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][i] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < HS; ++j) l_part[j] = 0.f;

    for (int cs = 0; cs < U0.nst; ++cs) {
      const int slot = g_comp % S;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], (g_comp / S) & 1, p.err));
      if (!ok) break;
      const uint8_t *kt = wbase + slot * G::kStageBytes;
      const uint8_t *vt = kt + G::kTileBytes;
      const int nvalid = min(16, U0.tok_end - (U0.tok_begin + cs * 16));

      // ---------------- scores (log2 units)
      float s[HS];
      if constexpr (HPC >= 4) {
        float2 sacc[2][HPC];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int h = 0; h < HPC; ++h) sacc[i][h] = make_float2(0.f, 0.f);
        constexpr int CPQ = D / 32;  // 8-element chunks per quarter of head_dim
#pragma unroll
        for (int cl = 0; cl < CPQ; ++cl) {
          float2 kf[2][4];
          load8<KV, D>(kt, t8, dq * CPQ + cl, kf[0]);
          load8<KV, D>(kt, t8 + 8, dq * CPQ + cl, kf[1]);
#pragma unroll
          for (int dpi = 0; dpi < 4; ++dpi) {
            const float4 *qp = reinterpret_cast<const float4 *>(q_s) + ((cl * 4 + dpi) * (HPC / 2)) * 4 + dq;
#pragma unroll
            for (int k = 0; k < HPC / 2; ++k) {
              const float4 qv = qp[k * 4];
              const float2 qa = make_float2(qv.x, qv.y), qb = make_float2(qv.z, qv.w);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                sacc[i][2 * k] = ffma2(kf[i][dpi], qa, sacc[i][2 * k]);
                sacc[i][2 * k + 1] = ffma2(kf[i][dpi], qb, sacc[i][2 * k + 1]);
              }
            }
          }
        }
        // reduce over the four quarters of head_dim
        float w[HPC];
        const bool odd_tok = dq & 1, hi_heads = dq >> 1;
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          const float v0 = sacc[0][h].x + sacc[0][h].y, v1 = sacc[1][h].x + sacc[1][h].y;
          const float keep = odd_tok ? v1 : v0, send = odd_tok ? v0 : v1;
          w[h] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int j = 0; j < HS; ++j) {
          const float keep = hi_heads ? w[HS + j] : w[j], send = hi_heads ? w[j] : w[HS + j];
          s[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
          s[j] = my_t < nvalid ? s[j] : kNegInf;
        }
      } else {
        float2 sacc = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int cc = 0; cc < D / 16; ++cc) {
          const int c = hh * (D / 16) + cc;
          float2 kf[4];
          load8<KV, D>(kt, my_t, c, kf);
          const float4 *qp = reinterpret_cast<const float4 *>(q_s + c * 8);
          const float4 qa = qp[0], qb = qp[1];
          sacc = ffma2(kf[0], make_float2(qa.x, qa.y), sacc);
          sacc = ffma2(kf[1], make_float2(qa.z, qa.w), sacc);
          sacc = ffma2(kf[2], make_float2(qb.x, qb.y), sacc);
          sacc = ffma2(kf[3], make_float2(qb.z, qb.w), sacc);
        }
        float x = sacc.x + sacc.y;
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        s[0] = my_t < nvalid ? x : kNegInf;
      }

      // ---------------- lazy online softmax: shuffles only when a score
      // exceeds the reference maximum by more than kRescaleLog2
      float mh[HS];
#pragma unroll
      for (int j = 0; j < HS; ++j) mh[j] = HPC >= 4 && (dq >> 1) ? m_ref[(HS + j) % HPC] : m_ref[j];
      bool over = false;
#pragma unroll
      for (int j = 0; j < HS; ++j) over |= s[j] > mh[j] + kRescaleLog2;
      if (__any_sync(0xffffffffu, over)) {
        float mx[HS], ms[HPC];
#pragma unroll
        for (int j = 0; j < HS; ++j) {
          mx[j] = s[j];
          if constexpr (HPC >= 4) {  // tokens live on t8 (lane bits 0-2) and dq bit 0 (lane bit 3)
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
            ms[j] = __shfl_sync(0xffffffffu, mx[j], 0);
            ms[HS + j] = __shfl_sync(0xffffffffu, mx[j], 16);
          } else {
#pragma unroll
            for (int off = 1; off < 16; off <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
            ms[0] = __shfl_sync(0xffffffffu, mx[0], 0);
          }
        }
        float alpha[HPC];
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          const float mn = fmaxf(m_ref[h], ms[h]);
          alpha[h] = fast_exp2(m_ref[h] - mn);
          m_ref[h] = mn;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[h][i].x *= alpha[h];
            acc[h][i].y *= alpha[h];
          }
        }
#pragma unroll
        for (int j = 0; j < HS; ++j) {
          const bool hi = HPC >= 4 && (dq >> 1);
          l_part[j] *= hi ? alpha[(HS + j) % HPC] : alpha[j];
          mh[j] = hi ? m_ref[(HS + j) % HPC] : m_ref[j];
        }
      }
      {
        float pv[HS];
#pragma unroll
        for (int j = 0; j < HS; ++j) {
          pv[j] = my_t < nvalid ? fast_exp2(s[j] - mh[j]) : 0.f;
          l_part[j] += (HPC >= 4 || hh == 0) ? pv[j] : 0.f;
        }
        if constexpr (HPC >= 4) {
          float4 *pw = reinterpret_cast<float4 *>(p_s + my_t * HPC + my_h0);
#pragma unroll
          for (int j2 = 0; j2 < HS / 2; ++j2)
            pw[j2] = make_float4(pv[2 * j2], pv[2 * j2], pv[2 * j2 + 1], pv[2 * j2 + 1]);
        } else if (hh == 0) {
          p_s[my_t] = make_float2(pv[0], pv[0]);
        }
      }
      __syncwarp();

      // ---------------- P.V
      {
        const int ts = lane / G::kLPT, dc = lane % G::kLPT;
        auto pv_step = [&](int t2) {
          float2 vf[4];
          load8<KV, D>(vt, t2, dc, vf);
          if constexpr (HPC >= 2) {
            const float4 *pp = reinterpret_cast<const float4 *>(p_s + t2 * HPC);
#pragma unroll
            for (int h2 = 0; h2 < HPC / 2; ++h2) {
              const float4 pq = pp[h2];
              const float2 pa = make_float2(pq.x, pq.y), pb = make_float2(pq.z, pq.w);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                acc[2 * h2][i] = ffma2(pa, vf[i], acc[2 * h2][i]);
                acc[2 * h2 + 1][i] = ffma2(pb, vf[i], acc[2 * h2 + 1][i]);
              }
            }
          } else {
            const float2 pa = p_s[t2];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[0][i] = ffma2(pa, vf[i], acc[0][i]);
          }
        };
        if (nvalid == 16) {  // full tile: straight-line, loads can be hoisted
#pragma unroll
          for (int k = 0; k < 16 / G::kTPS; ++k) pv_step(k * G::kTPS + ts);
        } else {  // ragged last tile: rows past the sequence end are never read
#pragma unroll
          for (int k = 0; k < 16 / G::kTPS; ++k)
            if (k * G::kTPS + ts < nvalid) pv_step(k * G::kTPS + ts);
        }
      }
      __syncwarp();  // this warp is done with the slot and with p_s
      ++g_comp;
      if (!have_next) {
        have_next = claim_step<HPC>(pc, U1, p, total_units, lane);
        if (have_next && U1.valid) issue_q(U1);
      }
      fill();
    }
    if (!ok) break;
    while (!have_next) {
      have_next = claim_step<HPC>(pc, U1, p, total_units, lane);
      if (have_next && U1.valid) issue_q(U1);
    }

    // ---------------- finish the unit
#pragma unroll
    for (int j = 0; j < HS; ++j)
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], off);
    float l_all[HPC];
#pragma unroll
    for (int j = 0; j < HS; ++j) {
      l_all[j] = __shfl_sync(0xffffffffu, l_part[j], 0);
      if constexpr (HPC >= 4) l_all[HS + j] = __shfl_sync(0xffffffffu, l_part[j], 16);
    }
#pragma unroll
    for (int off = G::kLPT; off < 32; off <<= 1)
#pragma unroll
      for (int h = 0; h < HPC; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[h][i].x += __shfl_xor_sync(0xffffffffu, acc[h][i].x, off);
          acc[h][i].y += __shfl_xor_sync(0xffffffffu, acc[h][i].y, off);
        }
    const int ts = lane / G::kLPT, dc = lane % G::kLPT;
    const int64_t head0 = (int64_t)U0.row * p.num_q_heads + U0.h0;
    if (U0.nparts == 1) {
      if (ts == 0) {
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          const float om = p.v_hs ? p.out_mult * __ldg(p.v_hs + U0.kvh) : p.out_mult;
          const float inv = l_all[h] > 0.f ? om / l_all[h] : 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t idx = (head0 + h) * D + dc * 8 + 2 * i;
            store_out<QT>(p.out, idx, p.out_f32 != 0, acc[h][i].x * inv);
            store_out<QT>(p.out, idx + 1, p.out_f32 != 0, acc[h][i].y * inv);
          }
        }
      }
    } else {
      if (ts == 0) {
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          float4 *dst = reinterpret_cast<float4 *>(
              p.ws_acc + ((head0 + h) * p.max_partitions + U0.part) * D + dc * 8);
          dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
          dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
        }
      }
      if (lane < HPC) {
        float mv = m_ref[0], lv = l_all[0];
#pragma unroll
        for (int h = 1; h < HPC; ++h)
          if (lane == h) {
            mv = m_ref[h];
            lv = l_all[h];
          }
        p.ws_ml[(head0 + lane) * p.max_partitions + U0.part] = make_float2(mv, lv);
      }
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        last = atomicAdd(p.ws_count + head0, 1) == U0.nparts - 1;
        if (last) p.ws_count[head0] = 0;  // ready for the next call
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        // lane q holds partition q's (max, sum); the warp reduces the weights,
        // then every lane combines D/32 output elements with independent loads
        constexpr int EPL = D / 32;  // output elements per lane
        for (int h = 0; h < HPC; ++h) {
          const int64_t base = (head0 + h) * p.max_partitions;
          float M = kNegInf;
          for (int q0 = 0; q0 < U0.nparts; q0 += 32) {
            const float mq = q0 + lane < U0.nparts ? __ldcg(&p.ws_ml[base + q0 + lane].x) : kNegInf;
            M = fmaxf(M, mq);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
          float a[EPL], l = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) a[e] = 0.f;
          for (int q0 = 0; q0 < U0.nparts; q0 += 32) {
            float wq = 0.f;
            if (q0 + lane < U0.nparts) {
              const float2 ml = __ldcg(&p.ws_ml[base + q0 + lane]);
              wq = fast_exp2(ml.x - M);
              l += wq * ml.y;
            }
            const int nq = min(32, U0.nparts - q0);
            for (int q = 0; q < nq; ++q) {
              const float w = __shfl_sync(0xffffffffu, wq, q);
              const float *src = p.ws_acc + (base + q0 + q) * D + lane * EPL;
              if constexpr (EPL == 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                a[0] += w * v.x; a[1] += w * v.y; a[2] += w * v.z; a[3] += w * v.w;
              } else {
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                a[0] += w * v.x; a[1] += w * v.y;
              }
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
          const float om = p.v_hs ? p.out_mult * __ldg(p.v_hs + U0.kvh) : p.out_mult;
          const float inv = l > 0.f ? om / l : 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            store_out<QT>(p.out, (head0 + h) * D + lane * EPL + e, p.out_f32 != 0, a[e] * inv);
        }
      }
    }

    // advance: U1 becomes current; the issue target follows it
    U0 = U1;
    U1.valid = 0;
    if (it_which == 1) it_which = 0;
    else set_target(U0, 0);
    fill();
  }
  // a warp that gave up on a timed-out wait still has copies in flight: let
  // them land (bounded) before the CTA's shared memory is released
  if (!ok) {
    for (uint32_t g = g_comp; g < g_issue; ++g) (void)mbar_wait(&full[g % S], (g / S) & 1, p.err);
  }
}

// Host launcher: plan kernel, then one persistent CTA per SM.
template <typename KV, typename QT, int D, int HPC>
cudaError_t launch_decode_one(const DecodeParams &p, const PoolMaps &m, cudaStream_t s) {
  using DG = DecGeo<KV, D, HPC>;
  decode_plan_kernel<0><<<1, 1024, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = paged_decode_kernel<KV, QT, D, HPC>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DG::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  kern<<<sms, DG::kNW * 32, DG::kSmem, s>>>(p, m.k, m.v);
  return cudaGetLastError();
}

template <typename KV, typename QT>
cudaError_t launch_decode(const DecodeParams &p, int hpc, const PoolMaps &m, int head_dim,
                          cudaStream_t s) {
  if (head_dim == 128) {
    if (hpc == 8) return launch_decode_one<KV, QT, 128, 8>(p, m, s);
    if (hpc == 4) return launch_decode_one<KV, QT, 128, 4>(p, m, s);
    return launch_decode_one<KV, QT, 128, 1>(p, m, s);
  }
  if (hpc == 8) return launch_decode_one<KV, QT, 64, 8>(p, m, s);
  if (hpc == 4) return launch_decode_one<KV, QT, 64, 4>(p, m, s);
  return launch_decode_one<KV, QT, 64, 1>(p, m, s);
}

}  // namespace pa
