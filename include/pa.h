/*
 * pa.h -- C ABI of libpa, a PagedAttention hot path for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the problem statement of these pages:
 *   [V07]  "Inside vLLM v0.7: How PagedAttention & Chunked Prefill Scaled 10x
 *          Token Serving" (bicarait.com)
 *   [ARCH] "Inside vLLM Architecture: How PagedAttention and Continuous
 *          Batching Solved the KV Cache Crisis" (codebumble.net)
 *   [HT]   "High-Throughput LLM Serving with vLLM & PagedAttention: Production
 *          Architecture & Optimization" (infoisland)
 *
 * Data model.  The KV cache of one attention layer is two pools, K and V, each
 * laid out [num_blocks][num_kv_heads][block_size][head_dim] in the element
 * type of the cache.  A sequence's token at position p lives in physical block
 * block_table[p / block_size] at offset p % block_size ([V07] "Architectural
 * Blueprint 2: How PagedAttention Actually Works"; [ARCH] "The Block Table
 * Mapping Subsystem").  Each (block, head) row group is one contiguous run of
 * block_size * head_dim elements.  A "slot" is block * block_size + offset.
 *
 * Conventions for every call:
 *  - Every pointer argument is DEVICE memory owned by the caller, except the
 *    pa_kv_cache descriptor, which is read on the host during the call.  The
 *    library allocates no memory and keeps no state between calls other than a
 *    per-device error word (see pa_get_device_error).
 *  - Calls are asynchronous: they validate arguments on the host, enqueue
 *    kernels on `stream` and return.  No call synchronises, except
 *    pa_get_device_error.  NULL stream = the legacy default stream.
 *  - Device pointers must be 16-byte aligned; q, out and the K/V inputs are
 *    contiguous [tokens or sequences][heads][head_dim] unless a stride is given.
 *  - Supported: head_dim 64 or 128; block_size 16 or 32; cache dtype f16,
 *    bf16 or fp8-e4m3; query dtype f16 or bf16 (equal to the cache dtype
 *    unless the cache is fp8).  Other combinations return PA_ERR_UNSUPPORTED.
 *  - Zero work (num_tokens, num_seqs, num_chunks or num_pairs == 0) returns
 *    PA_OK without launching anything.
 *  - Device-resident metadata (block ids, slots, sequence lengths) is the
 *    caller's contract.  The kernels check it as they read it: an out-of-range
 *    value is recorded in the device error word and the offending work is
 *    skipped; nothing traps.
 *  - A failed launch returns PA_ERR_CUDA.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points stay visible when the library is built with hidden visibility. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

/* Same type as the CUDA runtime's cudaStream_t, declared without CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative count, bad shape */
    PA_ERR_UNSUPPORTED = 2,  /* head_dim / block_size / dtype combination not built */
    PA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    PA_ERR_DEVICE_CHECK = 4, /* a kernel found out-of-range device metadata */
    PA_ERR_TIMEOUT = 5,      /* a kernel's bounded wait on an async copy expired */
    PA_ERR_NO_BLOCKS = 6     /* block manager: not enough free blocks for the request */
} pa_status;

/* PA_F32 is accepted only as the dtype of an attention output. */
typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2, PA_F32 = 3 } pa_dtype;

/* Shape and element type of one layer's K and V pools. */
typedef struct {
    int64_t num_blocks;   /* physical blocks in each pool */
    int32_t block_size;   /* tokens per block: 16 or 32 */
    int32_t num_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
    pa_dtype kv_dtype;    /* PA_F16, PA_BF16 or PA_FP8_E4M3 */
    /* fp8 only: one fp32 scale per pool; a stored code c means c * scale.
     * Ignored for f16/bf16 pools.  Must be finite and > 0 for fp8. */
    float k_scale;
    float v_scale;
    /* fp8 only, optional: device fp32 [num_kv_heads], one scale per KV head
     * (4-byte aligned, each finite and > 0, not checked on the device).  When
     * set, KV head h's codes mean c * k_head_scales[h] (resp. v_head_scales[h])
     * in every call and k_scale / v_scale are not used.  NULL: the per-pool
     * scale.  Must be NULL for f16/bf16 pools.  (Per-head scales are this
     * library's extension of the pages' per-tensor fp8 cache.) */
    const float *k_head_scales;
    const float *v_head_scales;
} pa_kv_cache;

/*
 * pa_reshape_and_cache -- scatter new tokens' K and V into their cache slots.
 *
 * Defined by the slot arithmetic of PagedKVCacheManager.allocate_slot ([ARCH]
 * "The Block Table Mapping Subsystem"): for every token t with
 * s = slot_mapping[t] >= 0 and every KV head h,
 *     k_cache[s / block_size][h][s % block_size][:] = k[t][h][:]   (same for v).
 * A negative slot marks a padding token and is skipped.
 *
 *   k, v          device, dtype in_dtype (PA_F16 or PA_BF16); token t, head h,
 *                 element e at index t * token_stride + h * head_dim + e
 *   token_stride  elements between consecutive tokens (>= num_kv_heads*head_dim,
 *                 a multiple of 8), so k and v may be views into a fused QKV
 *   slot_mapping  device int64 [num_tokens]
 *   k_cache, v_cache  device pools described by *cache
 * An f16/bf16 pool must have kv_dtype == in_dtype and receives the bits
 * unchanged.  An fp8 pool receives e4m3(fp32(x) / scale): IEEE fp32 division,
 * then round to nearest even with saturation to +-448 ([HT] "4. Production
 * vLLM Docker Deployment with FP8 Quantization", --kv-cache-dtype fp8; the
 * format and the per-tensor scale are this library's reading).
 * Slots >= num_blocks * block_size set PA_ERR_DEVICE_CHECK in the error word.
 * Two tokens mapping to the same slot race (the result is one of them).
 */
PA_API pa_status pa_reshape_and_cache(const void *k, const void *v, pa_dtype in_dtype,
                               int32_t num_tokens, int64_t token_stride,
                               const int64_t *slot_mapping, void *k_cache,
                               void *v_cache, const pa_kv_cache *cache,
                               pa_stream_t stream);

/*
 * pa_copy_blocks -- copy-on-write of shared blocks ([HT] "2. Virtual Memory
 * Paging Applied to GPUs: PagedAttention": when branches that share prompt
 * blocks diverge, a new block is allocated for the writer).
 *
 * For each pair i, the whole physical block src = pairs[2i] (every head, slot
 * and element) of both pools is copied bit for bit to dst = pairs[2i+1].
 *   src_dst_pairs  device int32 [num_pairs][2]
 * Destinations must be distinct and must not appear as a source in the same
 * call (pairs run in parallel).  Ids outside [0, num_blocks) set
 * PA_ERR_DEVICE_CHECK and that pair is skipped.
 */
PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const pa_kv_cache *cache,
                         const int32_t *src_dst_pairs, int32_t num_pairs,
                         pa_stream_t stream);

/*
 * pa_decode_workspace_bytes -- device workspace pa_decode needs: a work list
 * of (sequence, partition) items built on the device each call, and, when a
 * sequence can span several partitions, the split-KV partial results.
 *
 * partition_size 0 selects the library default (512 tokens); larger values
 * are treated as 512.  Returns 0 for invalid arguments (which pa_decode then
 * reports).
 */
PA_API size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_seq_len, int32_t partition_size);

/*
 * pa_decode -- paged attention for one query token per sequence (the decode
 * step; [V07] "Architectural Blueprint 3: Chunked Prefill", decode phase;
 * [ARCH] "Architectural Anatomy" pipeline: the kernel gathers the
 * non-contiguous K/V blocks while computing Q K^T).
 *
 * For sequence i with L = seq_lens[i] tokens (including the token being
 * decoded, whose K/V must already be in the cache) and query head h, reading
 * KV head g = h / (num_q_heads / num_kv_heads):
 *     out[i][h] = sum_p softmax_p(scale * q[i][h] . K_i[p][g]) * V_i[p][g]
 * over p = 0 .. L-1, where K_i[p] is the row at slot p % block_size of block
 * block_tables[i][p / block_size].  Exact attention ([ARCH] "Semantic FAQ
 * Section": paging does not change the result); fp32 accumulation.  L == 0
 * yields a zero row.  For an fp8 cache, K and V elements are code * scale.
 *
 *   q              device [num_seqs][num_q_heads][head_dim], dtype q_dtype
 *   block_tables   device int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens       device int32 [num_seqs], each <= max_seq_len and
 *                  <= max_blocks_per_seq * block_size
 *   max_seq_len    host upper bound of seq_lens; sizes the grid
 *   partition_size 0 = default (512); else a multiple of 32 tokens (values
 *                  above 512 act as 512).  A sequence longer than one
 *                  partition is split across workers and the pieces are
 *                  merged with a log-sum-exp combine.
 *   workspace      device, >= pa_decode_workspace_bytes(...) bytes, 256-byte
 *                  aligned.  Its contents on entry are ignored (each call
 *                  rebuilds them), so one workspace serves every call on a
 *                  stream; calls that may overlap need separate workspaces.
 *   out            device [num_seqs][num_q_heads][head_dim]
 *   out_dtype      q_dtype (rounded to nearest even from the fp32 result) or
 *                  PA_F32 (the fp32 result itself)
 */
PA_API pa_status pa_decode(const void *q, pa_dtype q_dtype, int32_t num_seqs,
                    int32_t num_q_heads, const void *k_cache,
                    const void *v_cache, const pa_kv_cache *cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *seq_lens, int32_t max_seq_len, float scale,
                    int32_t partition_size, void *workspace,
                    size_t workspace_bytes, void *out, pa_dtype out_dtype,
                    pa_stream_t stream);

/*
 * pa_decode_write -- one decode step in one call: the cache write of the
 * step's new tokens (pa_reshape_and_cache) fused with pa_decode.  Sequence i's
 * new token, row i of k_new / v_new, is stored at slot_mapping[i] exactly as
 * pa_reshape_and_cache stores it, and then every sequence attends exactly as
 * pa_decode does, the new token included ([V07] "Architectural Blueprint 3:
 * Chunked Prefill", decode phase: each step appends one token per sequence and
 * reads the whole cache).  With the tensor-core decode the token is stored by
 * the decode launch itself, before the work unit that reads it starts copying
 * its tiles; otherwise the cache write is launched first, on the same stream.
 *
 *   k_new, v_new   device [num_seqs][num_kv_heads][head_dim] in q_dtype, token
 *                  (row) stride token_stride elements (>= Hkv * head_dim, a
 *                  multiple of 8), 16-byte aligned
 *   slot_mapping   device int64 [num_seqs]: the slot of position seq_lens[i]-1
 *                  of sequence i (its last token), or negative for a sequence
 *                  with no new token this step.  Any other slot is a
 *                  violation: PA_ERR_DEVICE_CHECK may be recorded and the token
 *                  not stored.
 *   all other arguments as for pa_decode.
 */
PA_API pa_status pa_decode_write(const void *q, pa_dtype q_dtype, int32_t num_seqs,
                          int32_t num_q_heads, const void *k_new, const void *v_new,
                          int64_t token_stride, const int64_t *slot_mapping,
                          void *k_cache, void *v_cache, const pa_kv_cache *cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *seq_lens, int32_t max_seq_len, float scale,
                          int32_t partition_size, void *workspace,
                          size_t workspace_bytes, void *out, pa_dtype out_dtype,
                          pa_stream_t stream);

/*
 * pa_set_decode_kernel -- choose which of the library's two decode kernels
 * pa_decode and pa_decode_noalloc launch from now on (process-wide, any
 * thread, effective from the next call).  The pages describe one decode
 * kernel on CUDA cores; the choice is this library's own.  Both compute the
 * result defined above, in fp32, within the decode tolerance of each other.
 *   PA_DECODE_KERNEL_AUTO (default): the tensor-core kernel where it applies
 *     (head_dim 128 with 1 to 16 query heads per KV head, or head_dim 64
 *     with 1 to 8, any cache dtype, except one query head per KV head with
 *     a 16-bit cache: the Q.K^T and P.V of a KV head's query group run as
 *     MMAs, the group padded to 4, 8 or 16 rows),
 *     the CUDA-core kernel for every other shape;
 *   PA_DECODE_KERNEL_CUDA_CORES: the CUDA-core kernel for every shape.
 * Returns PA_ERR_INVALID_ARG for any other value (the setting is unchanged).
 */
typedef enum {
  PA_DECODE_KERNEL_AUTO = 0,
  PA_DECODE_KERNEL_CUDA_CORES = 1
} pa_decode_kernel;
PA_API pa_status pa_set_decode_kernel(int32_t kernel);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this call; it exists for the
 * library's users.
 *
 * Some callers cannot call cudaMalloc (or any allocator) at the point where
 * they decode: code that runs while allocation is forbidden or unsafe, such
 * as a host thread driving a memory pool that is fully carved up in advance,
 * or a runtime whose device memory is owned by another framework.  This entry
 * point takes the same arguments as pa_decode minus the workspace and uses a
 * fixed scratch area that lives inside the library: a static device array of
 * PA_NOALLOC_SCRATCH_BYTES (64 MiB).  Every GPU that loads the library holds
 * that array until the process exits.
 *
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress, a runtime call that
 *    allocates nothing).  The address is kept per device together with the
 *    id of the context it belongs to; after a cudaDeviceReset the next call
 *    sees a new context and looks the address up again.
 *  - A problem whose workspace (pa_decode_workspace_bytes) exceeds the array
 *    returns PA_ERR_UNSUPPORTED before anything is launched.
 *  - Every call on a device shares the one array.  Its contents are rebuilt
 *    by each call (the work list and counters are reset on the device before
 *    use), but two calls that overlap on the GPU (different streams without
 *    ordering) race on it and give undefined results.
 *  - No allocation of any kind is made; results equal pa_decode's.
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
PA_API pa_status pa_decode_noalloc(const void *q, pa_dtype q_dtype, int32_t num_seqs,
                            int32_t num_q_heads, const void *k_cache,
                            const void *v_cache, const pa_kv_cache *cache,
                            const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                            int32_t max_seq_len, float scale,
                            int32_t partition_size, void *out,
                            pa_dtype out_dtype, pa_stream_t stream);

/*
 * pa_prefill_chunk -- causal attention of prompt chunks over paged context
 * ([V07] "Architectural Blueprint 3: Chunked Prefill"; [HT] "5. Chunked
 * Prefill & Latency SLA Management": a long prompt is processed in chunks,
 * e.g. 512 tokens, batched with decodes).
 *
 * Chunk c owns query rows cu_q_lens[c] .. cu_q_lens[c+1]-1.  Row r of chunk c
 * sits at absolute position q_start[c] + r of sequence c and attends to
 * positions 0 .. q_start[c] + r inclusive, read through block_tables[c]:
 *     out[row][h] = sum_p softmax_p(scale * q[row][h] . K_c[p][g]) * V_c[p][g].
 * The chunk's own K/V must already be in the cache (pa_reshape_and_cache), so
 * seq_lens[c] must equal q_start[c] + (cu_q_lens[c+1] - cu_q_lens[c]).
 *
 *   q_chunk    device [total_q][num_q_heads][head_dim], total_q = cu_q_lens[num_chunks]
 *   cu_q_lens  device int32 [num_chunks + 1], non-decreasing, cu_q_lens[0] = 0
 *   q_start    device int32 [num_chunks]
 *   max_q_len  host upper bound of any chunk length; sizes the grid
 *   max_seq_len host upper bound of seq_lens
 *   out        device [total_q][num_q_heads][head_dim], dtype out_dtype
 *              (q_dtype or PA_F32, as for pa_decode)
 */
PA_API pa_status pa_prefill_chunk(const void *q_chunk, pa_dtype q_dtype,
                           const int32_t *cu_q_lens, const int32_t *q_start,
                           int32_t num_chunks, int32_t max_q_len,
                           int32_t num_q_heads, const void *k_cache,
                           const void *v_cache, const pa_kv_cache *cache,
                           const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *seq_lens,
                           int32_t max_seq_len, float scale, void *out,
                           pa_dtype out_dtype, pa_stream_t stream);

/*
 * pa_mixed_step -- one layer's chunked-prefill batch and decode batch in one
 * call ([V07] "Architectural Blueprint 3: Chunked Prefill": prompt chunks are
 * batched with decoding sequences; [HT] "5. Chunked Prefill & Latency SLA
 * Management").  The results are exactly those of pa_prefill_chunk on the
 * prefill part and of pa_decode_write (pa_decode when decode->k_new is null)
 * on the decode part, with the shared arguments below.  Where both parts run
 * on the tensor cores (head_dim 128, 4 or 8 query heads per KV head, the
 * default decode kernel) they share one launch after the decode's plan
 * kernel: the prefill chunks' tiles and the decode's persistent CTAs form one
 * grid, so the tensor-bound and the bandwidth-bound work run side by side.
 * Otherwise the decode and then the prefill are launched on the stream, as the
 * two calls would launch them.
 *
 * The parts must not meet in the cache: the prefill chunks' own K/V must
 * already be stored (as for pa_prefill_chunk), and no prefill chunk may read
 * a block that a decode row's new token is written into.
 *
 *   decode   the decode part; num_seqs 0 for none.  Fields as the arguments
 *            of pa_decode_write of the same names; k_new, v_new and
 *            slot_mapping all null for no new tokens.
 *   prefill  the prefill part; num_chunks 0 for none.  Fields as the
 *            arguments of pa_prefill_chunk of the same names.
 *   q_dtype, num_q_heads, k_cache, v_cache, cache, scale, out_dtype, stream:
 *            shared by both parts, as for those calls.
 * Errors: as those calls return them; nothing is launched when an argument
 * of either part is invalid.
 */
typedef struct {
  const void *q;                /* [num_seqs][num_q_heads][head_dim] */
  int32_t num_seqs;
  const int32_t *block_tables;  /* [num_seqs][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;
  const int32_t *seq_lens;      /* [num_seqs] */
  int32_t max_seq_len;
  int32_t partition_size;
  const void *k_new;            /* [num_seqs][num_kv_heads][head_dim], or null */
  const void *v_new;
  int64_t token_stride;
  const int64_t *slot_mapping;  /* [num_seqs], or null */
  void *workspace;              /* >= pa_decode_workspace_bytes(...) */
  size_t workspace_bytes;
  void *out;                    /* [num_seqs][num_q_heads][head_dim] */
} pa_decode_part;

typedef struct {
  const void *q_chunk;          /* [total_q][num_q_heads][head_dim] */
  const int32_t *cu_q_lens;     /* [num_chunks + 1] */
  const int32_t *q_start;       /* [num_chunks] */
  int32_t num_chunks;
  int32_t max_q_len;
  const int32_t *block_tables;  /* [num_chunks][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;
  const int32_t *seq_lens;      /* [num_chunks] */
  int32_t max_seq_len;
  void *out;                    /* [total_q][num_q_heads][head_dim] */
} pa_prefill_part;

PA_API pa_status pa_mixed_step(const pa_decode_part *decode, const pa_prefill_part *prefill,
                        pa_dtype q_dtype, int32_t num_q_heads, void *k_cache,
                        void *v_cache, const pa_kv_cache *cache, float scale,
                        pa_dtype out_dtype, pa_stream_t stream);

/*
 * pa_get_device_error -- read and clear the current device's error word.
 * Synchronises `stream`, then stores into *code the first device-side status
 * recorded since the last clear (PA_OK if none): PA_ERR_DEVICE_CHECK for
 * out-of-range metadata, PA_ERR_TIMEOUT for an expired wait.
 */
PA_API pa_status pa_get_device_error(pa_stream_t stream, int32_t *code);

/*
 * pa_selftest_wait_timeout -- check that the library's waits end.  The pages
 * have no counterpart; this call exists for the library's users and tests.
 *
 * Launches one warp that waits, with the same bounded wait every kernel of the
 * library uses, on an mbarrier that nothing completes.  The wait gives up
 * after its limit (about one second of %globaltimer), records PA_ERR_TIMEOUT
 * in the device error word (read it with pa_get_device_error) and the kernel
 * returns; the context stays usable.  Returns PA_ERR_CUDA if the launch fails.
 */
PA_API pa_status pa_selftest_wait_timeout(pa_stream_t stream);

/*
 * Block manager -- host-side bookkeeping of the paged pool (no GPU work, no
 * device memory): the block tables, slots and copy-on-write pairs that the
 * calls above take.  ([ARCH] "The Block Table Mapping Subsystem"; [V07]
 * "Architectural Blueprint 2: How PagedAttention Actually Works"; [HT] "2.
 * Virtual Memory Paging Applied to GPUs": blocks on demand, sharing with
 * reference counts, copy-on-write of a shared block on the first write.)
 *
 * A manager owns num_blocks physical blocks of block_size slots.  Sequences
 * are small integer ids it hands out.  A token at position p of a sequence
 * lives in slot table[p / block_size] * block_size + p % block_size.
 *  - pa_bm_create: shuffle_seed 0 hands out blocks in increasing id order; any
 *    other value hands them out in a seeded random order (a fragmented pool).
 *    *bm receives the manager, released with pa_bm_destroy.
 *  - pa_bm_new_sequence: an empty sequence.
 *  - pa_bm_fork: a new sequence sharing every block of `parent` (its length
 *    and table), e.g. one branch of parallel sampling.
 *  - pa_bm_append: extend `seq` by num_tokens positions; slots[i] (host
 *    int64, num_tokens entries) receives the slot of each new token, to pass
 *    to pa_reshape_and_cache.  A block is taken when a sequence enters a new
 *    logical block.  If the last block is shared (a fork) and partly filled,
 *    it is first replaced by a fresh copy: the (src, dst) block pair goes to
 *    cow_pairs (host int32, 2 per pair, cow_capacity pairs) and *num_cow
 *    receives the count (at most 1); run pa_copy_blocks on them before the
 *    cache write.  token_ids (host int32, num_tokens entries, or NULL) enables
 *    prefix reuse: every block this call fills completely is remembered by a
 *    hash of the token ids of the sequence up to and including it, and a later
 *    append that fills a block with the same ids after the same prefix shares
 *    that block instead of taking a new one; its slots are returned as -1,
 *    which pa_reshape_and_cache skips.  PA_ERR_NO_BLOCKS if the free blocks
 *    cannot cover the worst case (no reuse); PA_ERR_INVALID_ARG with *num_cow
 *    = 1 if a copy is needed and cow_capacity is 0.  Nothing changes on error.
 *  - pa_bm_free: release the sequence's blocks (a shared block returns to the
 *    free list when its last sequence releases it).
 *  - pa_bm_block_table: copy the sequence's table into `table` (host int32,
 *    `capacity` entries); *num_blocks and *seq_len receive its size and length
 *    (set even when capacity is too small, which returns PA_ERR_INVALID_ARG).
 *  - pa_bm_get_stats: pool occupancy.
 * Not thread-safe: one manager per thread, or external locking.
 */
typedef struct pa_block_manager pa_block_manager;
typedef struct {
    int32_t free_blocks;      /* blocks on the free list */
    int32_t used_blocks;      /* blocks with at least one reference */
    int32_t shared_blocks;    /* blocks referenced by more than one sequence */
    int32_t cached_blocks;    /* full blocks remembered for prefix reuse */
    int32_t live_sequences;
    int64_t logical_tokens;   /* sum of live sequences' lengths */
    int64_t logical_blocks;   /* sum of live sequences' table sizes */
} pa_bm_stats;

PA_API pa_status pa_bm_create(int32_t num_blocks, int32_t block_size,
                              uint64_t shuffle_seed, pa_block_manager **bm);
PA_API void pa_bm_destroy(pa_block_manager *bm);
PA_API pa_status pa_bm_new_sequence(pa_block_manager *bm, int32_t *seq);
PA_API pa_status pa_bm_fork(pa_block_manager *bm, int32_t parent, int32_t *child);
PA_API pa_status pa_bm_append(pa_block_manager *bm, int32_t seq, int32_t num_tokens,
                              const int32_t *token_ids, int64_t *slots,
                              int32_t *cow_pairs, int32_t cow_capacity,
                              int32_t *num_cow);
PA_API pa_status pa_bm_free(pa_block_manager *bm, int32_t seq);
PA_API pa_status pa_bm_block_table(const pa_block_manager *bm, int32_t seq,
                                   int32_t *table, int32_t capacity,
                                   int32_t *num_blocks, int32_t *seq_len);
PA_API pa_status pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *stats);

/* Static, human-readable name of a status code. */
PA_API const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
