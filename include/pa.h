/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged KV-cache library.
 *
 * PagedAttention keeps each sequence's K/V cache in fixed-size physical blocks
 * of block_size tokens and reaches them through a per-sequence block table
 * (CS349E Lecture 7 notes "KV Cache Management", §4.1; Month 2 · PagedAttention,
 * infra learning path, §5.2). The pages name three fused GPU operations around
 * it (CS349E Lecture 7 notes, §4.3): writing new tokens' K/V into their slots,
 * attention that reads through the block table, and one batched copy of the
 * blocks that copy-on-write duplicates. This header exposes those operations,
 * plus a split (partitioned) variant of the attention for long contexts.
 *
 * Conventions for every call:
 *   - Every pointer argument is device memory owned by the caller, unless the
 *     argument says "host". The library allocates nothing and keeps no pointer
 *     after a call returns.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream); the
 *     status they return reports argument checks and launch errors only.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and launches
 *     nothing.
 *   - Values that live in device memory (block ids, slots, context lengths,
 *     copy pairs) are checked by the kernels: an out-of-range value is skipped
 *     (never dereferenced) and recorded in a device error word that
 *     pa_get_error() reads. The kernels never trap.
 *   - Layouts are dense and row-major. A KV pool is HND,
 *     cache[num_blocks][num_kv_heads][block_size][head_dim], or NHD,
 *     cache[num_blocks][block_size][num_kv_heads][head_dim] (pa_kv_layout);
 *     token t of a sequence lives in physical block block_table[t / block_size],
 *     row t % block_size. Query head h reads kv head h / (num_heads / num_kv_heads).
 *   - q, out, key, value and the caches must be 16-byte aligned.
 *   - Supported: head_dim 64, 128 or 256; block_size 16 or 32; num_heads /
 *     num_kv_heads from 1 to 8; element types PA_F32, PA_F16, PA_BF16, and
 *     E4M3 caches through the *_fp8 calls (copy and swap move any type).
 *     The E4M3 decode calls take head_dim 128 and pa_decode_cascade head_dim
 *     64 or 128; other values return PA_ERR_UNSUPPORTED.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative or inconsistent size */
  PA_ERR_UNSUPPORTED = 2, /* valid but outside what this build implements */
  PA_ERR_OUT_OF_RANGE = 3, /* (pa_get_error) a device-side value was out of range */
  PA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  PA_ERR_NO_BLOCKS = 5     /* (block manager) no free physical block is left */
} pa_status;

/* Element types. PA_FP8_E4M3 is a cache-only type: one byte per element, an
 * E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448) read as code * scale with
 * one fp32 scale per K or V tensor. */
typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* KV pool layouts, the two the pages name (Month 2 · PagedAttention, infra
 * learning path, §5.2):
 *   PA_LAYOUT_HND  cache[num_blocks][num_kv_heads][block_size][head_dim]
 *   PA_LAYOUT_NHD  cache[num_blocks][block_size][num_kv_heads][head_dim]
 * A whole block is contiguous in both, so pa_copy_blocks and pa_swap_blocks
 * take no layout. An invalid value returns PA_ERR_INVALID_ARG. */
typedef enum { PA_LAYOUT_HND = 0, PA_LAYOUT_NHD = 1 } pa_kv_layout;

/* Bits of the device error word returned by pa_get_error(). */
#define PA_DEVERR_BLOCK_ID 1u /* a block-table entry outside [0, num_blocks) was skipped */
#define PA_DEVERR_SLOT 2u     /* a slot outside [-1, num_blocks * block_size) was skipped */
#define PA_DEVERR_CONTEXT 4u  /* a context length < 0 or beyond the table / workspace was clamped */
#define PA_DEVERR_PAIR 8u     /* a copy pair with an id outside [0, num_blocks) was skipped */
#define PA_DEVERR_TIMEOUT 16u /* an internal wait ran past its limit; the results are undefined (below) */
#define PA_DEVERR_PAIR_ALIAS 32u /* a copy / swap pair racing with another pair was skipped (see pa_copy_blocks) */

/*
 * Write each new token's K and V into the cache slot the block manager chose
 * for it (CS349E Lecture 7 notes §4.1 and §4.3: the slot is a row of a physical
 * block; CMU 15-779 Lecture 16 notes §3.3: new tokens fill the last block).
 *
 *   key, value    [num_tokens][num_kv_heads][head_dim], element type `dtype`
 *   k_cache,
 *   v_cache       pools of `dtype` in `layout` (HND or NHD, see pa_kv_layout)
 *   slot_mapping  int64 [num_tokens]; token t goes to block slot / block_size,
 *                 row slot % block_size; a negative slot means "skip" (padding)
 *
 * The copy is bit-exact. Slots must be distinct (two tokens writing the same
 * slot race). Slots >= num_blocks * block_size are skipped and recorded.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks,
                               pa_dtype dtype, cudaStream_t stream);

/*
 * Decode attention over a paged KV cache: for every sequence s and query head h
 * (Month 2 · PagedAttention §2.1 and §5.4; CS349E Lecture 7 notes §4.2)
 *
 *   out[s][h] = sum_{t < context_lens[s]} softmax_t(scale * q[s][h] . K_s[t]) V_s[t]
 *
 * with K_s[t] = k_cache[block_tables[s][t / block_size]][h / group][t % block_size]
 * (HND; NHD swaps the last two indices before head_dim) and group =
 * num_heads / num_kv_heads. Both layouts give bit-identical results.
 *
 *   out           [num_seqs][num_heads][head_dim], element type `out_dtype`
 *                 (`dtype` or PA_F32; accumulation is always fp32)
 *   q             [num_seqs][num_heads][head_dim], `dtype`
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; only the first
 *                 ceil(context_lens[s] / block_size) entries of a row are read
 *   context_lens  int32 [num_seqs]; the new token is included (it must already
 *                 be in the cache). 0 gives an all-zero output row.
 *
 * Context lengths beyond max_blocks_per_seq * block_size are clamped and recorded.
 */
pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                    pa_kv_layout layout, int64_t num_blocks, float scale, pa_dtype dtype, pa_dtype out_dtype,
                    cudaStream_t stream);

/*
 * Workspace size for pa_decode_split: with P = max(1, ceil(max_context_len /
 * partition_tokens)), it holds
 *   o  float [num_seqs][num_heads][P][head_dim]   normalised partial outputs
 *   m  float [num_seqs][num_heads][P]             partition max score, base-2 units
 *                                                 (scale * q . k * log2(e))
 *   l  float [num_seqs][num_heads][P]             sum of 2^(score - m) over the partition
 * each section starting on a 256-byte boundary, in that order. Returns 0 for
 * invalid sizes.
 */
size_t pa_decode_split_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                       int partition_tokens);

/*
 * Decode attention for long contexts, in two launches on `stream`:
 *   1. every (sequence, kv head, partition of partition_tokens tokens) is an
 *      independent work item that writes its partition's softmax statistics and
 *      normalised partial output into `workspace` (layout above);
 *   2. a reduce kernel merges the partitions of each (sequence, head) with
 *      log-sum-exp weights: M = max_p m_p, w_p = l_p 2^(m_p - M),
 *      out = sum_p w_p o_p / sum_p w_p -- the merge rule under which blockwise
 *      attention equals attention over the whole context (CMU 15-779 Lecture 16
 *      notes §3.3).
 * Arguments as pa_decode, plus:
 *   max_context_len   host int >= every context length (sizes the workspace;
 *                     longer contexts are clamped and recorded)
 *   partition_tokens  a positive multiple of block_size
 *   workspace         device scratch of at least workspace_bytes =
 *                     pa_decode_split_workspace_bytes(...), 16-byte aligned,
 *                     owned by the caller; its contents on entry are ignored and
 *                     after return hold the partition results
 * num_seqs may be at most 2048.
 */
pa_status pa_decode_split(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int max_blocks_per_seq,
                          const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                          int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks, float scale,
                          pa_dtype dtype, pa_dtype out_dtype, int max_context_len, int partition_tokens,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Size of the scratch array built into the library for pa_decode_split_static:
 * 16 MiB of device memory, held on every GPU that loads the library until the
 * process exits.
 */
#define PA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* PA_STATIC_SCRATCH_BYTES as the library was built (for bindings that cannot
 * read the macro). Host only; no CUDA call. */
size_t pa_static_scratch_bytes(void);

/*
 * pa_decode_split without a workspace argument. The pages have no counterpart
 * to this call: it exists for callers that cannot allocate device memory at
 * the point they run attention -- for example a plugin whose host framework
 * owns every device allocation and does not let it call cudaMalloc, or a
 * serving loop that must stay out of the CUDA allocator (which can synchronise
 * the device) once it is running. It computes exactly what pa_decode_split
 * computes, with the same arguments minus `workspace` / `workspace_bytes`, and
 * keeps the partition results in a scratch array of PA_STATIC_SCRATCH_BYTES
 * inside the library instead. It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 *   - Arguments are checked exactly as pa_decode_split checks them (same
 *     statuses), then the size limit:
 *     pa_decode_split_workspace_bytes(num_seqs, num_heads, head_dim,
 *     max_context_len, partition_tokens) must not exceed
 *     PA_STATIC_SCRATCH_BYTES (e.g. 8 sequences x 64 heads x head_dim 128 fit
 *     up to 63 partitions, 32,256 tokens at 512-token partitions); a larger
 *     request returns PA_ERR_UNSUPPORTED and launches nothing -- use
 *     pa_decode_split with a workspace for it.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture. With CUDA's lazy module loading (the default) that first
 *     call can also be when the driver loads the library's device code and
 *     commits the array's 16 MiB, so the "allocates nothing" guarantee holds
 *     from the second call on: make one call (or any pa_* call that launches a
 *     kernel) during set-up, outside the region that must not allocate.
 *   - The address is cached per device for the life of the process; do not
 *     use the library across cudaDeviceReset() (the same holds for the error
 *     word every call reports into).
 *   - Every call, on every stream, shares the one array and leaves its
 *     contents behind: calls whose executions overlap on the GPU race and give
 *     undefined results. Nothing in the array needs to start at zero.
 */
pa_status pa_decode_split_static(void* out, const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int block_size, pa_kv_layout layout, int64_t num_blocks,
                                 float scale, pa_dtype dtype, pa_dtype out_dtype, int max_context_len,
                                 int partition_tokens, cudaStream_t stream);

/*
 * Decode attention for batches whose sequences share prompt prefixes (parallel
 * samples of one prompt, a common system prompt): sequences
 * [group_starts[g], group_starts[g+1]) share their first prefix_lens[g] tokens
 * through the same physical blocks (CS349E Lecture 7 notes §5.1 and §5.3).
 * The result equals pa_decode's; attention over a context is the merge of
 * attention over any split of it (CMU 15-779 Lecture 16 notes §3.3), so it is
 * computed in three launches:
 *   1. prefix pass: each (group, kv head, partition of the prefix) attends all
 *      of the group's query rows at once, so a prefix block is read once per
 *      group instead of once per member (groups of more than 16 query rows run
 *      it on tcgen05 tensor cores, M = 64 or 128 rows per tile);
 *   2. each sequence's own tokens [prefix, context) as one partial per
 *      (sequence, head), one warp per (sequence, kv head), longest first;
 *   3. the log-sum-exp reduce of both.
 * Arguments as pa_decode_split, plus (device int32 arrays):
 *   group_starts  [num_groups + 1], group_starts[0] = 0, non-decreasing,
 *                 group_starts[num_groups] = num_seqs (every sequence in one group)
 *   prefix_lens   [num_groups]; rounded down to whole blocks; must not exceed any
 *                 member's context length (violations are clamped and recorded)
 *   max_group_size     host int >= every group's size; max_group_size *
 *                      (num_heads / num_kv_heads) <= 128
 *   max_prefix_len     host int >= every prefix_lens[g] (a longer prefix_lens[g],
 *                      or one past the block table's width, is clamped to
 *                      what the workspace and table hold and recorded as
 *                      PA_DEVERR_CONTEXT)
 *   max_context_len    host int >= every context length
 * The tokens of a group's prefix are read through the block table of its
 * first member. 16-bit caches only; num_seqs and num_groups at most 2048.
 * Workspace: pa_decode_cascade_workspace_bytes(...) bytes, laid out as for
 * pa_decode_split with P = ceil(max_prefix_len / T) + 1 slots (the prefix
 * partitions, then one slot for each sequence's own tokens; max_context_len is
 * accepted for symmetry with pa_decode_split and bounds nothing), followed by
 * num_seqs x 6 bytes (256-byte aligned) where the prefix pass leaves the
 * suffix pass its schedule. Its contents need no initialisation.
 */
size_t pa_decode_cascade_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_prefix_len,
                                         int max_context_len, int partition_tokens);

pa_status pa_decode_cascade(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                            pa_kv_layout layout, int64_t num_blocks, float scale, pa_dtype dtype,
                            pa_dtype out_dtype, const int32_t* group_starts, const int32_t* prefix_lens, int num_groups,
                            int max_group_size, int max_prefix_len, int max_context_len, int partition_tokens,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Batched copy-on-write block copies (CS349E Lecture 7 notes §5.1 and §4.3: a
 * sample about to write into a shared block first gets its own copy; all copies
 * pending for a step go in one launch). For every pair p and every layer l:
 *   k_caches[l][block_pairs[p][1]] = k_caches[l][block_pairs[p][0]]   (all heads, rows)
 *   v_caches[l][block_pairs[p][1]] = v_caches[l][block_pairs[p][0]]
 *
 *   k_caches, v_caches  HOST arrays of num_layers device pointers, each a pool
 *                       [num_blocks][num_kv_heads][block_size][head_dim] of `dtype`
 *                       (or NHD: the copy moves whole blocks, contiguous in both)
 *   block_pairs         int64 [num_pairs][2] (src, dst)
 *
 * The copy is bit-exact. All pairs are copied in parallel, so destinations must
 * be distinct and no destination may also be a source (its own pair's or
 * another's). The kernel checks this on the device: every pair whose
 * destination is another pair's destination or any pair's source, or whose
 * source is another pair's destination, is skipped in every layer (neither K
 * nor V is written) and PA_DEVERR_PAIR_ALIAS is recorded; the other pairs are
 * copied. Pairs with an id outside [0, num_blocks) are skipped and recorded as
 * PA_DEVERR_PAIR (and race with nothing). The check reads the whole pair list
 * once per CTA, which is small next to the blocks for the few hundred pairs of
 * a decode step; it grows as num_pairs^2.
 */
pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                         const int64_t* block_pairs, int num_pairs, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, pa_dtype dtype, cudaStream_t stream);

/*
 * FP8 KV cache (E4M3 codes with one fp32 scale for K and one for V). Keeping
 * the cache in 8 bits is one of the ways the pages list to make KV smaller
 * (CS349E Lecture 7 notes, §10 and §11); it halves the bytes every decode step
 * reads. Reading taken: element value = decode(code) * k_scale (or v_scale).
 *
 * pa_reshape_and_cache_fp8: as pa_reshape_and_cache, but key and value (of
 * `in_dtype`: PA_F32, PA_F16 or PA_BF16) are quantised on the way in:
 * code = E4M3(x / scale), the division in fp32 (correctly rounded), then round
 * to nearest even on the E4M3 grid; finite values beyond +-448 saturate, NaN
 * stays NaN. k_cache / v_cache hold codes in `layout`.
 *
 * pa_decode_fp8 / pa_decode_split_fp8: as pa_decode / pa_decode_split over an
 * E4M3 cache: out = softmax(scale * q . (k_scale * K)) (v_scale * V). q is of
 * `q_dtype` (PA_F16 or PA_BF16) and is converted to fp16 inside the kernel
 * (exact for |q| in [2^-14, 65504]); out is `q_dtype` or PA_F32. head_dim must
 * be 128. The split variant uses the workspace layout of pa_decode_split.
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* k_cache, void* v_cache,
                                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                                   int block_size, pa_kv_layout layout, int64_t num_blocks, pa_dtype in_dtype,
                                   float k_scale, float v_scale, cudaStream_t stream);

pa_status pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        pa_kv_layout layout, int64_t num_blocks, float scale, float k_scale, float v_scale,
                        pa_dtype q_dtype, pa_dtype out_dtype, cudaStream_t stream);

pa_status pa_decode_split_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                              pa_kv_layout layout, int64_t num_blocks, float scale, float k_scale, float v_scale,
                              pa_dtype q_dtype, pa_dtype out_dtype, int max_context_len, int partition_tokens, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * Move KV blocks between two pools in one launch: the GPU <-> CPU swap of
 * preempted sequences (CS349E Lecture 7 notes §6.2: a preempted sequence's
 * blocks go to CPU memory and come back later; done as per-block copies each
 * layer's K and V cost layers x 2 x blocks small transfers with a fixed
 * overhead each). For every pair p and every layer l:
 *   dst_k_caches[l][block_pairs[p][1]] = src_k_caches[l][block_pairs[p][0]]  (same for V)
 *
 *   dst_*_caches, src_*_caches  HOST arrays of num_layers pool pointers; a pool
 *                               is [*_num_blocks][num_kv_heads][block_size][head_dim]
 *                               of `dtype`, in device memory or in pinned host
 *                               memory (cudaHostAlloc / cudaMallocHost), which
 *                               the kernel reads or writes directly at its host
 *                               address (unified addressing)
 *   block_pairs                 int64 [num_pairs][2] (src id, dst id), device
 *                               memory or pinned host memory
 *
 * Bit-exact. Destinations must be distinct; checked on the device as for
 * pa_copy_blocks (a pair whose destination is another pair's destination is
 * skipped and recorded as PA_DEVERR_PAIR_ALIAS). Where a layer's source and
 * destination pool are the same memory (the same pointer), ids of both sides
 * name the same blocks and the copy-on-write rule applies in full: no
 * destination may be any pair's source. Pools that overlap without being the
 * same pointer are not supported. Ids outside their pool are skipped and
 * recorded (PA_DEVERR_PAIR).
 */
pa_status pa_swap_blocks(void* const* dst_k_caches, void* const* dst_v_caches,
                         const void* const* src_k_caches, const void* const* src_v_caches, int num_layers,
                         const int64_t* block_pairs, int num_pairs, int num_kv_heads, int head_dim,
                         int block_size, int64_t dst_num_blocks, int64_t src_num_blocks, pa_dtype dtype,
                         cudaStream_t stream);

/*
 * Read and clear the calling device's error word (PA_DEVERR_* bits) after the
 * work already queued on `stream` has finished. *error_bits (host) receives the
 * bits. Returns PA_ERR_OUT_OF_RANGE when any bit was set, PA_OK otherwise. It
 * synchronises `stream`.
 *
 * There is one error word per device, shared by every stream: the bits read
 * are those set by any of the library's kernels that ran on the device since
 * the last read, on whatever stream; kernels of other streams still running
 * may set bits after the read. To attribute bits to one stream, synchronise
 * the device's other streams first (or use one stream).
 */
pa_status pa_get_error(uint32_t* error_bits, cudaStream_t stream);

/*
 * PA_DEVERR_TIMEOUT: every wait inside a kernel (on the arrival of its own TMA
 * copies or tensor-core results) gives up after 2 s of wall time instead of
 * spinning forever; the kernel then stops, lets its copies in flight land and
 * returns, and the CUDA context stays usable. On a healthy GPU these waits
 * last microseconds, so the bit means the GPU was starved (time-sliced with
 * other work, preempted for seconds) or faulty. The outputs of the launches
 * that ran since the last read of the error word are then undefined; nothing
 * else is: the attention calls only read the caches, and a copy or cache write
 * that stopped early wrote some of its rows. Re-issuing the same calls on the
 * same inputs recomputes them (cache writes and copies are idempotent for a
 * well-formed slot mapping and pair list).
 */

/*
 * pa_get_error without the bits: waits for `stream`, reads and clears the
 * calling device's error word, and returns PA_ERR_OUT_OF_RANGE if any bit was
 * set (PA_OK otherwise; PA_ERR_CUDA if a CUDA call failed). The device-side
 * range checks it reports are always compiled in, not only in debug builds.
 */
pa_status pa_debug_check(cudaStream_t stream);

/*
 * Diagnostic of the bounded waits that every kernel uses on its mbarriers
 * (each gives up after a time limit instead of spinning forever).
 *
 * Launches one CTA of two warps on `stream`. Warp 0 waits on an mbarrier that
 * nothing completes and gives up after limit_ns (host value, nanoseconds); it
 * raises the CTA's abort flag and ORs PA_DEVERR_TIMEOUT into the error word.
 * Warp 1 waits on a second such barrier with a limit 50 times longer and must
 * leave as soon as it sees the abort flag, as the decode kernels' warps do
 * once one of them has given up. The call therefore takes about limit_ns of
 * device time, not 50 times that, and leaves the CUDA context usable. Read the
 * result with pa_get_error().
 *
 * limit_ns must lie in [1000, 100000000] (1 us to 100 ms); otherwise
 * PA_ERR_INVALID_ARG, with no CUDA call. Asynchronous; allocates nothing.
 */
pa_status pa_check_wait_limit(uint64_t limit_ns, cudaStream_t stream);

/* A static, human-readable name for a status (never NULL). pa_status_str and
 * pa_status_string are the same function under two names. */
const char* pa_status_str(pa_status status);
const char* pa_status_string(pa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

/*
 * Host block manager (CPU only; no CUDA call). It produces the block tables,
 * slot mappings and copy-on-write pairs the kernels above consume:
 *   - a pool of num_blocks blocks of block_size tokens; a sequence gets a new
 *     block only when its last one is full (CS349E Lecture 7 notes §4.1);
 *   - fork shares blocks (reference counts); appending into a shared,
 *     partially filled last block copies it first and returns the pair
 *     (§5.1);
 *   - with prefix_caching != 0, each full block is keyed by a chain hash of
 *     (parent block's hash, its tokens), so only whole block-aligned prefixes
 *     match (Month 2 · PagedAttention §6.3, §7.5); a new sequence reuses the
 *     cached blocks of its longest matching prefix; a released block that holds
 *     a cached full block stays reusable until it is evicted, least recently
 *     released first, when no other free block is left (§7.2-§7.3; CS349E §8).
 * Not thread-safe: one manager per thread (or external locking).
 *
 * pa_bm_create         NULL on bad sizes or allocation failure.
 * pa_bm_add_sequence   prefill: blocks for tokens[0..num_tokens); *cached_tokens
 *                      (may be NULL) receives how many leading tokens came from
 *                      the prefix cache (a multiple of block_size). Unknown /
 *                      duplicate ids: PA_ERR_INVALID_ARG; pool exhausted:
 *                      PA_ERR_NO_BLOCKS (nothing is changed).
 * pa_bm_fork           child shares every block of parent.
 * pa_bm_append         reserve the slot of the sequence's next token (slot =
 *                      block * block_size + row); *cow_src / *cow_dst receive the
 *                      copy-on-write pair or -1.
 * pa_bm_free           release the sequence's blocks (tail first).
 * pa_bm_block_table    writes up to `capacity` block ids; returns the table
 *                      length, or -1 for an unknown sequence.
 * pa_bm_context_len    tokens of the sequence, or -1.
 * pa_bm_num_free       blocks available (free + evictable).
 * pa_bm_stats          out[6] = {prefix-cache block lookups, hits, evictions,
 *                      copy-on-write copies, evictable blocks, cached blocks}.
 */
typedef struct pa_bm pa_bm;
pa_bm* pa_bm_create(int64_t num_blocks, int block_size, int prefix_caching);
void pa_bm_destroy(pa_bm* bm);
pa_status pa_bm_add_sequence(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int32_t num_tokens,
                             int32_t* cached_tokens);
pa_status pa_bm_fork(pa_bm* bm, int64_t parent_id, int64_t child_id);
pa_status pa_bm_append(pa_bm* bm, int64_t seq_id, int32_t token, int64_t* slot, int64_t* cow_src,
                       int64_t* cow_dst);
pa_status pa_bm_free(pa_bm* bm, int64_t seq_id);
int32_t pa_bm_block_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int32_t capacity);
int64_t pa_bm_context_len(const pa_bm* bm, int64_t seq_id);
int64_t pa_bm_num_free(const pa_bm* bm);
void pa_bm_stats(const pa_bm* bm, int64_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
