// pa_attention.cuh -- paged attention on CUDA cores, one CTA per query row:
// the chunked-prefill path for shapes the tensor-core kernel does not take
// (head_dim 64, GQA groups outside {1, 2, 4, 8, 16}); each prefill row sees
// its own causal length.  The tile geometry (Geo), the swizzled tile reads
// (load8) and the output store are shared with the persistent decode
// (pa_decode.cuh).  With no cu_q_lens the kernel treats each row as a decode
// row of length seq_lens[row].
//
// What it computes ("Inside vLLM Architecture", sections "Architectural
// Anatomy: PagedAttention Virtual Memory Paging" and "CUDA Shared Memory
// Optimization in PagedAttention"; exactness: "Semantic FAQ Section"):
//   out[row][h] = sum_p softmax_p(scale * q[row][h] . K[p][g]) V[p][g],
// g = h / (Hq / Hkv), with K[p] / V[p] gathered from physical block
// table[p / bs], slot p % bs of the pools [num_blocks][Hkv][bs][D].
//
// How, on sm_103a:
//  * One CTA = (row, KV head, group of HPC query heads, token partition);
//    grid = (rows, KV heads x head groups, partitions).
//    The HPC heads of a GQA group share every K/V byte read from HBM.
//  * A producer warp walks the block table (32 entries per coalesced load)
//    and issues 2D bulk-tensor (TMA) copies of 16-token K and V tiles into
//    a ring of shared-memory slots, 128-byte swizzled, completion tracked by
//    mbarriers.  Four consumer warps take tiles round-robin; each warp owns
//    two ring slots, so its next tile is in flight while it computes.
//  * Q.K^T: one lane per (token, half of the heads), the whole head_dim in
//    registers -- no cross-lane reduction of the dot product; q (pre-scaled
//    by scale*log2 e) is broadcast from shared memory; packed fp32x2 FMAs.
//  * Online softmax per warp in the log2 domain (ex2), warp-shuffle maxima
//    ("partial softmax reductions" in the page's words); probabilities go
//    through a small per-warp shared buffer to the P.V mapping.
//  * P.V: one lane per 8 output elements, all HPC heads, packed FMAs.
//  * The four warps' states are merged in shared memory.  A row longer than
//    one partition is split over CTAs; each writes (acc, max, sum) to the
//    workspace and the last CTA to arrive (atomic counter, reset after use)
//    combines the partitions: out = sum_p 2^(m_p-M) acc_p / sum_p 2^(m_p-M) l_p.
//  * fp8-e4m3 KV: codes are widened in registers (e4m3 -> f16 -> f32, exact);
//    k_scale is folded into the q pre-scale, v_scale into the output.
//  * Metadata is checked as it is read (block ids, lengths); bad values set
//    the device error word and the work is skipped.  Every mbarrier wait is
//    bounded in time.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

template <typename KV, int D>
struct Geo {
  static constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  static constexpr int kEB = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kEB;                       // 256, 128 or 64
  static constexpr int kPanelBytes = kRowBytes < 128 ? kRowBytes : 128;
  static constexpr int kPanels = kRowBytes / kPanelBytes;
  static constexpr int kPanelElems = kPanelBytes / kEB;           // TMA box width
  static constexpr int kStageTok = 16;                            // TMA box height
  static constexpr int kPanelTileBytes = kStageTok * kPanelBytes;
  static constexpr int kTileBytes = kStageTok * kRowBytes;        // one of K / V
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kNW = 4;                                   // consumer warps
  static constexpr int kSlots = 2 * kNW;
  static constexpr int kThreads = (kNW + 1) * 32;
  static constexpr int kLPT = D / 8;                              // P.V lanes per token
  static constexpr int kTPS = 32 / kLPT;                          // P.V tokens per step
  static_assert(kPanelTileBytes % 1024 == 0 || kPanelBytes == 64, "swizzle atom alignment");
};

template <typename KV, int D, int HPC>
struct Smem {
  using G = Geo<KV, D>;
  static constexpr int kStagesOff = 0;
  static constexpr int kQOff = G::kSlots * G::kStageBytes;
  static constexpr int kPOff = kQOff + D * HPC * 4;
  static constexpr int kBarOff = kPOff + G::kNW * G::kStageTok * HPC * 8;
  static constexpr int kFlagOff = kBarOff + 2 * G::kSlots * 8;
  static constexpr int kBytes = kFlagOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
  // merge buffers alias the stage ring once every tile is consumed
  static constexpr int kMergeAcc = 0;
  static constexpr int kMergeM = G::kNW * HPC * D * 4;
  static constexpr int kMergeL = kMergeM + G::kNW * HPC * 4;
  static_assert(kMergeL + G::kNW * HPC * 4 <= kQOff, "merge buffers must fit in the ring");
};

// 8 consecutive elements [8c, 8c+8) of row t of a swizzled tile, widened to fp32 pairs.
template <typename KV, int D>
__device__ __forceinline__ void load8(const uint8_t *tile, int t, int c, float2 (&f)[4]) {
  using G = Geo<KV, D>;
  if constexpr (G::kFp8) {
    const uint32_t off = (uint32_t)t * G::kPanelBytes + (uint32_t)c * 8;
    const uint2 w = *reinterpret_cast<const uint2 *>(tile + swz<G::kPanelBytes>(off));
    f[0] = unpack2_e4m3(w.x);
    f[1] = unpack2_e4m3(w.x >> 16);
    f[2] = unpack2_e4m3(w.y);
    f[3] = unpack2_e4m3(w.y >> 16);
  } else {
    const int byte = c * 16;
    const int panel = byte / G::kPanelBytes;
    const uint32_t off = (uint32_t)t * G::kPanelBytes + (uint32_t)(byte % G::kPanelBytes);
    const uint4 w = *reinterpret_cast<const uint4 *>(tile + panel * G::kPanelTileBytes +
                                                     swz<G::kPanelBytes>(off));
    f[0] = unpack2(w.x, KV{});
    f[1] = unpack2(w.y, KV{});
    f[2] = unpack2(w.z, KV{});
    f[3] = unpack2(w.w, KV{});
  }
}

// Output element: fp32 as computed, or rounded to the query dtype.
template <typename QT>
__device__ __forceinline__ void store_out(void *out, int64_t idx, bool f32, float x) {
  if (f32) static_cast<float *>(out)[idx] = x;
  else static_cast<QT *>(out)[idx] = Elem<QT>::from_f32(x);
}

template <typename KV, typename QT, int D, int HPC>
__global__ void __launch_bounds__(Geo<KV, D>::kThreads)
    paged_attention_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                           const __grid_constant__ CUtensorMap tmap_v) {
  using G = Geo<KV, D>;
  using S = Smem<KV, D, HPC>;
  constexpr int NW = G::kNW;
  const float kNegInf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  float *q_s = reinterpret_cast<float *>(smem + S::kQOff);        // [D/2][HPC][2]
  float2 *p_s = reinterpret_cast<float2 *>(smem + S::kPOff);      // [NW][16][HPC]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOff);
  uint64_t *empty = full + G::kSlots;
  int *flag = reinterpret_cast<int *>(smem + S::kFlagOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gqa = p.num_q_heads / p.num_kv_heads;
  const int groups = gqa / HPC;
  const int kvh = blockIdx.y / groups;
  const int h0 = kvh * gqa + (blockIdx.y % groups) * HPC;
  const int part = blockIdx.z;
  const int bs = p.block_size;

  // ------------------------------------------------ row, length, table
  int row, L;
  const int32_t *table;
  if (p.cu_q_lens == nullptr) {
    row = blockIdx.x;
    L = __ldg(p.seq_lens + row);
    table = p.block_tables + (int64_t)row * p.max_blocks_per_seq;
  } else {
    const int c = blockIdx.x / p.max_q_len, r = blockIdx.x % p.max_q_len;
    const int c0 = __ldg(p.cu_q_lens + c), n = __ldg(p.cu_q_lens + c + 1) - c0;
    if (r >= n) return;
    row = c0 + r;
    const int qs = __ldg(p.q_start + c);
    L = qs + r + 1;
    if (tid == 0 && blockIdx.y == 0 && r == 0 && __ldg(p.seq_lens + c) != qs + n)
      record_error(p.err, PA_ERR_DEVICE_CHECK);
    table = p.block_tables + (int64_t)c * p.max_blocks_per_seq;
  }
  const int64_t cap = min((int64_t)p.max_blocks_per_seq * bs,
                          (int64_t)p.max_partitions * p.partition_size);
  if (L < 0 || L > cap) {
    if (tid == 0 && blockIdx.y == 0 && part == 0) record_error(p.err, PA_ERR_DEVICE_CHECK);
    L = L < 0 ? 0 : (int)cap;
  }
  const int nparts = (L + p.partition_size - 1) / p.partition_size;
  const int64_t out_row = ((int64_t)row * p.num_q_heads + h0) * D;  // element index
  const bool out_f32 = p.out_f32 != 0;
  if (L == 0) {
    if (part == 0)
      for (int e = tid; e < HPC * D; e += blockDim.x) store_out<QT>(p.out, out_row + e, out_f32, 0.f);
    return;
  }
  if (part >= nparts) return;
  const int tok_begin = part * p.partition_size;
  const int tok_end = min(L, tok_begin + p.partition_size);
  const int nst = (tok_end - tok_begin + G::kStageTok - 1) / G::kStageTok;

  // ------------------------------------------------ setup
  if (tid == 0) {
    for (int s = 0; s < G::kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == NW && lane == 0) {
    prefetch_tensor_map(&tmap_k);
    prefetch_tensor_map(&tmap_v);
  }
  {
    const QT *qrow = static_cast<const QT *>(p.q) + ((int64_t)row * p.num_q_heads + h0) * D;
    for (int e = tid; e < HPC * D; e += blockDim.x) {
      const int h = e / D, d = e % D;
      q_s[((d >> 1) * HPC + h) * 2 + (d & 1)] =
          Elem<QT>::to_f32(qrow[e]) * (p.k_hs ? p.q_mult * __ldg(p.k_hs + kvh) : p.q_mult);
    }
  }
  __syncthreads();

  float2 acc[HPC][4];
  float m_run[HPC];
  constexpr int HH = HPC >= 2 ? HPC / 2 : 1;
  float l_part[HH];
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    m_run[h] = kNegInf;
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[h][i] = make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int j = 0; j < HH; ++j) l_part[j] = 0.f;

  if (warp == NW) {
    // ============================================== producer warp
    int win = -1;
    int32_t my_blk = -1;
    for (int j = 0; j < nst; ++j) {
      const int tok = tok_begin + j * G::kStageTok;
      const int lblk = tok / bs;
      if ((lblk & ~31) != win) {
        win = lblk & ~31;
        const int li = win + lane;
        my_blk = li < p.max_blocks_per_seq ? __ldg(table + li) : -1;
      }
      const int32_t blk = __shfl_sync(0xffffffffu, my_blk, lblk - win);
      const int slot = j % G::kSlots;
      int ok = 1;
      if (lane == 0) {
        if (j >= G::kSlots) ok = mbar_wait(&empty[slot], ((j / G::kSlots) - 1) & 1, p.err);
        if (ok) {
          if (blk < 0 || blk >= p.num_blocks) {
            record_error(p.err, PA_ERR_DEVICE_CHECK);
            mbar_arrive(&full[slot]);
          } else {
            mbar_arrive_expect_tx(&full[slot], G::kStageBytes);
            const int32_t y = (blk * p.num_kv_heads + kvh) * bs + (tok % bs);
            uint8_t *st = smem + slot * G::kStageBytes;
#pragma unroll
            for (int pn = 0; pn < G::kPanels; ++pn) {
              tma_load_2d(st + pn * G::kPanelTileBytes, &tmap_k, &full[slot],
                          pn * G::kPanelElems, y);
              tma_load_2d(st + G::kTileBytes + pn * G::kPanelTileBytes, &tmap_v, &full[slot],
                          pn * G::kPanelElems, y);
            }
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else {
    // ============================================== consumer warps
    for (int j = warp; j < nst; j += NW) {
      const int slot = j % G::kSlots;
      const bool ok = mbar_wait(&full[slot], (j / G::kSlots) & 1, p.err);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t *kt = smem + slot * G::kStageBytes;
      const uint8_t *vt = kt + G::kTileBytes;
      const int nvalid = min(G::kStageTok, tok_end - (tok_begin + j * G::kStageTok));
      const int t = lane & 15, hh = lane >> 4;

      // ---------------- scores (log2 units): lane = (token t, head half hh)
      float s[HH];
      if constexpr (HPC >= 2) {
        float2 sacc[HH];
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) sacc[jh] = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          float2 kf[4];
          load8<KV, D>(kt, t, c, kf);
#pragma unroll
          for (int dp = 0; dp < 4; ++dp) {
            const float2 *qp = reinterpret_cast<const float2 *>(q_s) + (c * 4 + dp) * HPC + hh * HH;
#pragma unroll
            for (int jh = 0; jh < HH; ++jh) sacc[jh] = ffma2(kf[dp], qp[jh], sacc[jh]);
          }
        }
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) s[jh] = t < nvalid ? sacc[jh].x + sacc[jh].y : kNegInf;
      } else {
        // one head: the two half-warps split head_dim and add
        float2 sacc = make_float2(0.f, 0.f);
#pragma unroll 4
        for (int cc = 0; cc < D / 16; ++cc) {
          const int c = hh * (D / 16) + cc;
          float2 kf[4];
          load8<KV, D>(kt, t, c, kf);
#pragma unroll
          for (int dp = 0; dp < 4; ++dp)
            sacc = ffma2(kf[dp], reinterpret_cast<const float2 *>(q_s)[c * 4 + dp], sacc);
        }
        float x = sacc.x + sacc.y;
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        s[0] = t < nvalid ? x : kNegInf;
      }

      // ---------------- online softmax over this tile
      float ms[HPC];
      {
        float mx[HH];
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) {
          mx[jh] = s[jh];
#pragma unroll
          for (int off = 1; off < 16; off <<= 1)
            mx[jh] = fmaxf(mx[jh], __shfl_xor_sync(0xffffffffu, mx[jh], off));
        }
        if constexpr (HPC >= 2) {
#pragma unroll
          for (int jh = 0; jh < HH; ++jh) {
            const float other = __shfl_xor_sync(0xffffffffu, mx[jh], 16);
            ms[jh] = hh ? other : mx[jh];
            ms[HH + jh] = hh ? mx[jh] : other;
          }
        } else {
          ms[0] = mx[0];
        }
      }
      bool grow = false;
#pragma unroll
      for (int h = 0; h < HPC; ++h) grow |= ms[h] > m_run[h];
      if (grow) {  // warp-uniform: every lane holds the same ms and m_run
        float alpha[HPC];
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          const float mn = fmaxf(m_run[h], ms[h]);
          alpha[h] = fast_exp2(m_run[h] - mn);
          m_run[h] = mn;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[h][i].x *= alpha[h];
            acc[h][i].y *= alpha[h];
          }
        }
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) l_part[jh] *= (HPC >= 2 && hh) ? alpha[(HH + jh) % HPC] : alpha[jh];
      }
      {
        float2 *pw = p_s + (warp * G::kStageTok + t) * HPC;
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) {
          const float mh = (HPC >= 2 && hh) ? m_run[(HH + jh) % HPC] : m_run[jh];
          const float pv = t < nvalid ? fast_exp2(s[jh] - mh) : 0.f;
          if (HPC >= 2 || hh == 0) {
            l_part[jh] += pv;
            pw[(HPC >= 2 ? hh * HH : 0) + jh] = make_float2(pv, pv);
          }
        }
      }
      __syncwarp();

      // ---------------- P.V: lane = (token sub-step ts, 8-element chunk dc)
      {
        const int ts = lane / G::kLPT, dc = lane % G::kLPT;
#pragma unroll
        for (int k = 0; k < G::kStageTok / G::kTPS; ++k) {
          const int t2 = k * G::kTPS + ts;
          if (t2 < nvalid) {
            float2 vf[4];
            load8<KV, D>(vt, t2, dc, vf);
            const float2 *pp = p_s + (warp * G::kStageTok + t2) * HPC;
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
              const float2 ph = pp[h];
#pragma unroll
              for (int i = 0; i < 4; ++i) acc[h][i] = ffma2(ph, vf[i], acc[h][i]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    // reduce this warp's state across lanes
#pragma unroll
    for (int jh = 0; jh < HH; ++jh)
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) l_part[jh] += __shfl_xor_sync(0xffffffffu, l_part[jh], off);
#pragma unroll
    for (int off = G::kLPT; off < 32; off <<= 1)
#pragma unroll
      for (int h = 0; h < HPC; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[h][i].x += __shfl_xor_sync(0xffffffffu, acc[h][i].x, off);
          acc[h][i].y += __shfl_xor_sync(0xffffffffu, acc[h][i].y, off);
        }
  }

  // ------------------------------------------------ merge the warps
  __syncthreads();  // every tile consumed: the ring may be reused
  float *mg_acc = reinterpret_cast<float *>(smem + S::kMergeAcc);
  float *mg_m = reinterpret_cast<float *>(smem + S::kMergeM);
  float *mg_l = reinterpret_cast<float *>(smem + S::kMergeL);
  if (warp < NW) {
    const int ts = lane / G::kLPT, dc = lane % G::kLPT;
    if (ts == 0) {
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        float4 *dst = reinterpret_cast<float4 *>(mg_acc + (warp * HPC + h) * D + dc * 8);
        dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
        dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
      }
    }
    if ((lane & 15) == 0) {
      const int hh = lane >> 4;
      if (HPC >= 2 || hh == 0)
#pragma unroll
        for (int jh = 0; jh < HH; ++jh) mg_l[warp * HPC + (HPC >= 2 ? hh * HH : 0) + jh] = l_part[jh];
    }
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < HPC; ++h) mg_m[warp * HPC + h] = m_run[h];
  }
  __syncthreads();

  const bool split = nparts > 1;
  const int64_t ws_head = (int64_t)row * p.num_q_heads + h0;
  for (int e = tid; e < HPC * D; e += blockDim.x) {
    const int h = e / D, d = e % D;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mg_m[w * HPC + h]);
    float a = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mg_m[w * HPC + h];
      const float wt = mw == kNegInf ? 0.f : fast_exp2(mw - M);
      a += wt * mg_acc[(w * HPC + h) * D + d];
      l += wt * mg_l[w * HPC + h];
    }
    if (!split) {
      store_out<QT>(p.out, out_row + e, out_f32,
                    l > 0.f ? a / l * (p.v_hs ? p.out_mult * __ldg(p.v_hs + kvh) : p.out_mult) : 0.f);
    } else {
      const int64_t slot = (ws_head + h) * p.max_partitions + part;
      p.ws_acc[slot * D + d] = a;
      if (d == 0) p.ws_ml[slot] = make_float2(M, l);
    }
  }
  if (!split) return;

  // ------------------------------------------------ split-KV: last CTA combines
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(p.ws_count + ws_head, 1);
    const int last = prev == nparts - 1;
    if (last) p.ws_count[ws_head] = 0;  // leave the workspace zeroed for the next call
    *flag = last;
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  for (int e = tid; e < HPC * D; e += blockDim.x) {
    const int h = e / D, d = e % D;
    const int64_t base = (ws_head + h) * p.max_partitions;
    float M = kNegInf;
    for (int q = 0; q < nparts; ++q) M = fmaxf(M, __ldcg(&p.ws_ml[base + q].x));
    float a = 0.f, l = 0.f;
    for (int q = 0; q < nparts; ++q) {
      const float2 ml = __ldcg(&p.ws_ml[base + q]);
      const float wt = fast_exp2(ml.x - M);
      a += wt * __ldcg(&p.ws_acc[(base + q) * D + d]);
      l += wt * ml.y;
    }
    store_out<QT>(p.out, out_row + e, out_f32,
                  l > 0.f ? a / l * (p.v_hs ? p.out_mult * __ldg(p.v_hs + kvh) : p.out_mult) : 0.f);
  }
}

// Host launcher for one (KV storage, Q type): picks head_dim and heads-per-CTA.
template <typename KV, typename QT, int D, int HPC>
cudaError_t launch_one(const AttnParams &p, const PoolMaps &m, int rows, cudaStream_t s) {
  using Sm = Smem<KV, D, HPC>;
  auto kern = paged_attention_kernel<KV, QT, D, HPC>;
  // set on every launch: the attribute is per device, and cheap to set
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sm::kAlloc);
  if (e != cudaSuccess) return e;
  const int groups = (p.num_q_heads / p.num_kv_heads) / HPC;
  dim3 grid(rows, p.num_kv_heads * groups, p.max_partitions);
  kern<<<grid, Geo<KV, D>::kThreads, Sm::kAlloc, s>>>(p, m.k, m.v);
  return cudaGetLastError();
}

template <typename KV, typename QT>
cudaError_t launch_attention(const AttnParams &p, const PoolMaps &m, int head_dim, int rows,
                             cudaStream_t s) {
  const int hpc = p.heads_per_cta;
  if (head_dim == 128) {
    if (hpc == 8) return launch_one<KV, QT, 128, 8>(p, m, rows, s);
    if (hpc == 4) return launch_one<KV, QT, 128, 4>(p, m, rows, s);
    return launch_one<KV, QT, 128, 1>(p, m, rows, s);
  }
  if (hpc == 8) return launch_one<KV, QT, 64, 8>(p, m, rows, s);
  if (hpc == 4) return launch_one<KV, QT, 64, 4>(p, m, rows, s);
  return launch_one<KV, QT, 64, 1>(p, m, rows, s);
}

}  // namespace pa
