// pa_mixed_tc.cuh -- a chunked-prefill step and a decode step in one launch:
// the prefill chunks' tensor-core tiles and the decode's persistent CTAs in
// one grid, so that the tensor-bound prefill tiles and the bandwidth-bound
// decode share the GPU instead of running one after the other ("Inside vLLM
// v0.7", "Architectural Blueprint 3: Chunked Prefill": a batch mixes prompt
// chunks with decoding sequences; "High-Throughput LLM Serving with vLLM &
// PagedAttention", "5. Chunked Prefill & Latency SLA Management").
//
// What it computes: exactly what pa_prefill_chunk and pa_decode (or
// pa_decode_write) compute for the two parts; each block runs one of the two
// CTA bodies unchanged.  Blocks 0 .. P-1 are the prefill CTAs (one Q tile of
// 128 GQA-packed rows of one KV head each, the prefill kernel's grid laid out
// in a line); blocks P .. P+S-1 are the decode's persistent CTAs, S the SM
// count.  Blocks start in index order as SMs come free, so the prefill tiles
// start at once, the decode CTAs fill the remaining SMs and then each SM a
// prefill tile leaves; the decode work is claimed from one cursor, so decode
// CTAs that start late simply claim less of it.  The decode CTAs wait for the
// plan kernel (programmatic launch); the prefill CTAs do not.
//
// One CTA per SM (either body uses most of shared memory); the block is the
// decode body's twelve warps (four loaders, a merging warp), of which a
// prefill CTA uses the first nine.
#pragma once

#include "pa_decode_tc.cuh"
#include "pa_prefill_tc.cuh"

namespace pa {

// The block is the decode body's twelve warps (four loaders, a merging warp);
// a prefill CTA's body uses its first nine and the rest have no role.
constexpr int kMixedThreads = dtc::Roles::threads_for(4, true);

template <typename KV, typename QT, int G>
__global__ void __launch_bounds__(kMixedThreads, 1)
    mixed_tc_kernel(const DecodeTcParams tp, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const PrefillTcParams pp, int prefill_ctas,
                    int prefill_x) {
  static_assert(kMixedThreads >= tc::Roles<1>::kThreads, "the prefill roles fit in the block");
  const int b = blockIdx.x;   // block-uniform: every barrier of a body is reached by its whole block
  if (b < prefill_ctas) prefill_tc_body<KV, QT, G, 1>(pp, b % prefill_x, b / prefill_x, &tmap_k, &tmap_v);
  else decode_tc_body<KV, QT, G, 128, 4, true>(tp, &tmap_k, &tmap_v);
}

// Host launcher: the decode's plan kernel, then the mixed grid as its
// programmatic dependent.  pp.row_blocks is set here (one Q tile per CTA).
template <typename KV, typename QT, int G>
cudaError_t launch_mixed_tc_one(const DecodeTcParams &tp, const PoolMaps &m, const PrefillTcParams &pp0,
                                int num_chunks, cudaStream_t s) {
  constexpr bool kFp8 = std::is_same<KV, uint8_t>::value;
  constexpr bool kSplit = std::is_same<QT, __nv_bfloat16>::value && !kFp8;
  constexpr int smem_d = dtc::TcGeo<G, kSplit, kFp8, dtc::QTerms<KV, QT>::value>::kSmemBytes;
  constexpr int smem_p = tc::Layout<1, kFp8>::kSmemBytes;
  constexpr int smem = smem_d > smem_p ? smem_d : smem_p;
  constexpr int BR = tc::kM / G;   // token rows per prefill CTA
  PrefillTcParams pp = pp0;
  pp.row_blocks = (pp.max_q_len + BR - 1) / BR;
  const int64_t px = (int64_t)num_chunks * pp.row_blocks;
  const int64_t pctas = px * pp.num_kv_heads;
  int sms = 0;
  cudaError_t e = current_sm_count(&sms);
  if (e != cudaSuccess) return e;
  if (pctas + sms > 2147483647ll) return cudaErrorInvalidValue;
  if ((e = launch_decode_tc_plan(tp.d, tp.jobs, s)) != cudaSuccess) return e;
  if ((e = ensure_smem_limit<mixed_tc_kernel<KV, QT, G>>(smem)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(pctas + sms));
  cfg.blockDim = dim3(kMixedThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mixed_tc_kernel<KV, QT, G>, tp, m.k, m.v, pp, (int)pctas, (int)px);
}

template <typename KV, typename QT>
cudaError_t launch_mixed_tc(const DecodeTcParams &tp, const PoolMaps &m, const PrefillTcParams &pp, int num_chunks,
                            int gqa, cudaStream_t s) {
  switch (gqa) {
    case 4: return launch_mixed_tc_one<KV, QT, 4>(tp, m, pp, num_chunks, s);
    case 8: return launch_mixed_tc_one<KV, QT, 8>(tp, m, pp, num_chunks, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
