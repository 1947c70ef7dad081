/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged decode-attention library
 * (libpagedattn.so).
 *
 * Sources (web pages on LLM inference, cited by short tag):
 *   [QA]    "LLM推理与服务：面试问题与推荐回答" (LLM inference & serving interview Q&A)
 *   [SB11]  "Scaling Book 入门第 11 章：推理优化 — KV Cache / Continuous Batching / 量化"
 *   [H100]  "09-inference-optimization.md" (LLM-Code-Hot-100, "⚡ 推理优化")
 *   [ANIM]  "推理机制动态图解（进阶）：并行、投机解码、PD、FlashAttention、调度"
 *   [PANO]  "LLM 推理优化全景实战：从 PagedAttention 到投机解码"
 *
 * The KV cache of one attention layer is a pool of fixed-size physical blocks
 * ([QA] Q2; [PANO] §2.2-2.3).  Each sequence owns a block table mapping its
 * logical blocks to physical ones, like an operating-system page table.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers are DEVICE pointers on the current CUDA device; `stream` is a
 *    cudaStream_t passed as void* (NULL = legacy default stream).  Every call is
 *    asynchronous on `stream` and returns after the launch.
 *  - The caller owns every buffer.  The library allocates no device memory and
 *    keeps no per-call state; its device-resident state is one 32-bit error
 *    word per device (see pa_device_error) and the fixed workspace array of
 *    pa_decode_split_noalloc.
 *  - 16-bit floating point (fp16 or bf16, chosen by `dtype`) for q, K, V and the
 *    output; fp32 arithmetic inside.
 *  - Layouts (dense, row-major):
 *      k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *                        (per page and head, block_size consecutive token rows:
 *                        the [H100] PagedKVCache page shape
 *                        [layers, heads, page_size, head_dim] for one layer)
 *      q, out            [num_seqs][q_len][num_q_heads][head_dim]
 *      k_new, v_new      [n_tokens][num_kv_heads][head_dim]
 *      block_tables      int32 [num_seqs][max_blocks_per_seq]
 *      context_lens      int32 [num_seqs]
 *      slot_mapping      int64 [n_tokens]
 *  - Token position pos of sequence i lives in slot
 *      block_tables[i][pos / block_size] * block_size + pos % block_size
 *    ([PANO] §2.3 write_kv), i.e. block slot / block_size, row slot % block_size.
 *  - context_lens count this step's new tokens: append runs first, then
 *    attention, and a new token attends to itself ([H100] "KV Cache":
 *    AttentionWithKVCache.forward updates the cache before computing scores).
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads)
 *    (contiguous groups; [QA] Q7, [ANIM] §1 figure).
 *  - Supported now: block_size 8, 16 or 32 (the kernels walk 16-token tiles: a
 *    32-token block is two tiles, a tile of an 8-token pool spans two blocks);
 *    head_dim 64 or 128; q_len 1..4096 with a
 *    16-bit cache (up to 16 query rows per sequence go to the decode kernel, more
 *    to a tensor-core kernel that shares each K/V chunk among 128 query rows of a
 *    KV head: chunked prefill,
 *    [QA] Q14, [SB11] §11.3 "Continuous Batching"); q_len 1..4096 with an FP8
 *    cache too, split between the same two kernels (the many-row kernel widens
 *    each chunk of codes to fp16 in shared memory).
 *  - Alignment: every pointer 16-byte aligned.
 *
 * Errors: argument checks run on the host before any launch and return
 * PA_ERR_INVALID_ARG (null pointer, non-positive size, num_q_heads not a
 * multiple of num_kv_heads, misaligned pointer, workspace too small, sizes whose
 * indices overflow 32 bits) or PA_ERR_UNSUPPORTED (head_dim, block_size, q_len or
 * dtype outside the supported set).  A failed launch returns PA_ERR_CUDA.
 * Kernels never trap or assert: a block id outside [0, num_blocks) or a slot
 * outside the pool is skipped (attention reads zeros in its place) and sets
 * PA_ERR_DEVICE_CHECK in the device error word; a device-side wait that exceeds
 * about two seconds gives up and sets PA_ERR_DEVICE_TIMEOUT.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,
    PA_ERR_UNSUPPORTED = -2,
    PA_ERR_CUDA = -3,
    PA_ERR_DEVICE_CHECK = -4,
    PA_ERR_DEVICE_TIMEOUT = -5
} pa_status;

typedef enum { PA_FP16 = 0, PA_BF16 = 1 } pa_dtype;

/* Human-readable name of a status code (static string, never NULL). */
PA_API const char *pa_status_string(pa_status status);

/* Library ABI version (major * 100 + minor). */
PA_API int pa_version(void);

/*
 * pa_slot_mapping -- slots of this step's new tokens ([PANO] §2.3 write_kv:
 * logical_block = pos // block_size, block_offset = pos % block_size).
 * For sequence i the new tokens are its last q_len positions
 * pos = context_lens[i] - q_len + u (u = 0..q_len-1), written to
 * slot_mapping[i*q_len + u]; a position < 0 gives -1 (skipped by pa_append_kv).
 * A position whose logical block is >= max_blocks_per_seq gives -1 and sets
 * PA_ERR_DEVICE_CHECK.  slot_mapping: int64 [num_seqs*q_len], written.
 */
PA_API pa_status pa_slot_mapping(int64_t *slot_mapping, const int32_t *block_tables,
                                 const int32_t *context_lens, int num_seqs,
                                 int max_blocks_per_seq, int block_size, int q_len,
                                 void *stream);

/*
 * pa_append_kv -- scatter this step's new K/V rows into the pool
 * ([PANO] §2.3 write_kv; [H100] PagedKVCache.append_token).
 * Row t of k_new/v_new (all heads) is copied bit for bit to slot
 * slot_mapping[t]: block slot / block_size, row slot % block_size.  Slots < 0
 * are skipped; slots >= num_blocks*block_size are skipped and set
 * PA_ERR_DEVICE_CHECK.  Two tokens with the same slot: undefined which wins.
 * k_cache, v_cache: read-write.  n_tokens == 0 is a no-op.
 */
PA_API pa_status pa_append_kv(void *k_cache, void *v_cache, const void *k_new,
                              const void *v_new, const int64_t *slot_mapping, int n_tokens,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              pa_dtype dtype, void *stream);

/*
 * pa_copy_blocks -- copy-on-write support: sequences that share physical blocks
 * (parallel sampling, beam search, a cached prefix; [QA] Q2) keep sharing them
 * until one of them writes; before that write it needs a private copy.  For each
 * pair i, block src_blocks[i] (every head, every row, K and V) is copied bit for
 * bit to block dst_blocks[i].  Pairs with an id outside [0, num_blocks) are skipped
 * and set PA_ERR_DEVICE_CHECK.  A destination that is also a source or another
 * pair's destination in the same call: undefined result.  src_blocks, dst_blocks:
 * int32 [n_pairs] device arrays.  n_pairs == 0 is a no-op.
 */
PA_API pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_blocks,
                                const int32_t *dst_blocks, int n_pairs, int num_kv_heads,
                                int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                                void *stream);

/*
 * pa_decode -- attention of every query row over its sequence's paged K/V, in
 * one pass with online softmax ([ANIM] §5: running max m, running sum l,
 * unnormalised output rescaled by exp(m_old - m_new), output O / l at the end;
 * [PANO] §2.4 for what is computed: softmax(q K^T * scale) V over the gathered
 * blocks).  Only positions t < context_lens[i] are used ([H100]
 * PagedKVCache.get_kv keeps used_slots rows of the last page).  With q_len > 1,
 * query u of sequence i sees positions t <= context_lens[i] - q_len + u (the
 * [H100] causal mask triu(diagonal = Lk - Lq + 1)).  A row that sees no
 * position (context length 0) is written as zeros.
 * out: [num_seqs][q_len][num_q_heads][head_dim], written (round to nearest even).
 * The query heads of one GQA group share every K/V read.
 */
PA_API pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, float scale, void *stream,
                           int max_blocks_per_seq, int num_blocks, int q_len, pa_dtype dtype);

/*
 * Split-KV (flash-decoding, [SB11] §11.8): one sequence's blocks are cut into
 * num_splits partitions processed by different thread blocks, then merged.
 *
 * Workspace layout (fp32, caller-allocated, pa_decode_workspace_size bytes),
 * with R = q_len * num_q_heads rows per sequence (row u*num_q_heads + h):
 *   acc [num_seqs][num_splits][R][head_dim]   unnormalised sum_t 2^(s_t - m) V_t
 *   m   [num_seqs][num_splits][R]             max_t s_t  (-inf if empty)
 *   l   [num_seqs][num_splits][R]             sum_t 2^(s_t - m)  (0 if empty)
 * where s_t = scale * log2(e) * q.k_t (base-2 units).  Section m starts at
 * byte offset align256(sizeof acc), section l at align256 after m.
 * Partition p of sequence i covers blocks [p*C, (p+1)*C) with
 * C = ceil(ceil(context_lens[i] / block_size) / num_splits); partitions past
 * the end are empty.  With 8-token blocks the partitions are counted in 16-token
 * tiles instead (C = ceil(ceil(context_lens[i] / 16) / num_splits) tiles).
 */
PA_API size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int q_len, int head_dim,
                                       int num_splits);

/* Partial pass: writes every (sequence, partition, row) entry of the workspace. */
PA_API pa_status pa_decode_partial(void *workspace, size_t workspace_bytes, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, float scale, int num_splits,
                                   int max_blocks_per_seq, int num_blocks, int q_len,
                                   pa_dtype dtype, void *stream);

/*
 * Combine pass (the online-softmax rescale of [ANIM] §5 applied across
 * partitions): M = max_p m_p; out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p
 * over non-empty partitions; zeros if all are empty.  Reads the workspace,
 * writes out [num_seqs][q_len][num_q_heads][head_dim].
 */
PA_API pa_status pa_decode_combine(void *out, const void *workspace, size_t workspace_bytes,
                                   int num_seqs, int num_q_heads, int head_dim, int q_len,
                                   int num_splits, pa_dtype dtype, void *stream);

/*
 * pa_append_decode -- one decode step fused: slot mapping, append of the new K/V
 * rows and attention in one launch (a second launch, the combine, when
 * num_splits > 1).  Kernel fusion of consecutive memory-bound steps follows
 * [SB11] §11.8 ("Kernel Fusion").  Equivalent to pa_slot_mapping, then
 * pa_append_kv of k_new/v_new (rows [num_seqs*q_len][num_kv_heads][head_dim], the
 * last q_len positions of each sequence), then pa_decode (num_splits == 1;
 * workspace may be NULL) or pa_decode_partial + pa_decode_combine (num_splits > 1;
 * workspace as for pa_decode_partial).  The cache ends up bit-identical to the
 * unfused sequence and out within the same tolerance.  New positions < 0 are
 * skipped; new positions beyond the block table or the pool are skipped and set
 * PA_ERR_DEVICE_CHECK.  With q_len > 16 the append is a launch of its own before
 * the attention (a CTA's rows then depend on rows other CTAs would write).
 */
PA_API pa_status pa_append_decode(void *out, const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size, float scale,
                                  int max_blocks_per_seq, int num_blocks, int q_len,
                                  pa_dtype dtype, int num_splits, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * pa_decode_cascade -- attention of a batch whose sequences all begin with the
 * same prefix_blocks physical blocks (a shared prompt: [QA] Q2 copy-on-write page
 * sharing and Q3 prefix caching; [SB11] §11.4 "Prefix Caching": the shared
 * prefix's KV is stored once).  Same result as pa_append_decode, computed in
 * three launches over a workspace of 1 + tail_splits partitions
 * (pa_decode_workspace_size(num_seqs, num_q_heads, q_len, head_dim,
 * 1 + tail_splits) bytes, 256-byte aligned, layout as for pa_decode_partial):
 *   partition 0      every query row of every sequence against the prefix blocks,
 *                    read once per KV head for all num_seqs * q_len * group rows;
 *                    the prefix is the first prefix_blocks entries of block-table
 *                    row 0;
 *   partitions 1..   each sequence's blocks from prefix_blocks on (with this
 *                    step's append when k_new/v_new are given), cut into
 *                    tail_splits equal parts;
 * then the combine.  With tail_splits == 1 and q_len <= 16 the tail pass is a
 * single pass that merges partition 0 into its result (no combine launch).  It
 * runs alongside the prefix pass and waits for it only before that merge.  The
 * causal limit applies in both passes.
 * Caller's contract: for every sequence, table entries [0, prefix_blocks) equal
 * those of row 0, and this step's new tokens lie at or past position
 * prefix_blocks * block_size (so the append never writes a shared block).
 * prefix_blocks * block_size must be a multiple of 16 (PA_ERR_UNSUPPORTED
 * otherwise: the two passes split at a 16-token tile).
 * k_new and v_new are both NULL (no append) or both given.  16-bit caches only.
 */
PA_API pa_status pa_decode_cascade(void *out, const void *q, const void *k_new, const void *v_new,
                                   void *k_cache, void *v_cache, const int32_t *block_tables,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size, float scale,
                                   int max_blocks_per_seq, int num_blocks, int q_len,
                                   pa_dtype dtype, int prefix_blocks, int tail_splits,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * FP8 (e4m3) KV cache.  The pool holds one byte per element, same layout
 * [num_blocks][num_kv_heads][block_size][head_dim]; an element stands for
 * e4m3_value * scale[kv_head], with separate fp32 scales for K and V
 * (k_scale, v_scale: device arrays [num_kv_heads]).  Quantisation ([QA] Q4: KV
 * quantisation relieves KV memory; fewer bytes per token on a bandwidth-bound path)
 * is code = e4m3(x / scale): fp32 division, round to nearest even, magnitudes above
 * 448 saturate to 448.  head_dim 128 only.
 *
 * pa_append_kv_fp8 -- pa_append_kv for an FP8 cache: k_new/v_new are 16-bit rows of
 * type new_dtype, quantised as above into their slots.
 */
PA_API pa_status pa_append_kv_fp8(void *k_cache, void *v_cache, const void *k_new,
                                  const void *v_new, const int64_t *slot_mapping, int n_tokens,
                                  int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                  pa_dtype new_dtype, const float *k_scale, const float *v_scale,
                                  void *stream);

/*
 * pa_decode_fp8 -- attention over an FP8 cache (q and out of type dtype; fp32
 * arithmetic on the dequantised K, V).  With k_new/v_new (both non-NULL) the step's
 * new rows are first quantised into the cache as pa_append_kv_fp8 would (slots of
 * the last q_len positions, as pa_slot_mapping), in the same launch.  num_splits == 1:
 * single pass, workspace may be NULL; num_splits > 1: split-KV partial pass into the
 * workspace (layout of pa_decode_partial) and the combine.  With more than 16
 * query rows per sequence (chunked prefill over an FP8 cache, [QA] Q4 and Q14) the
 * fused append is a launch of its own before the attention, as in pa_append_decode.
 */
PA_API pa_status pa_decode_fp8(void *out, const void *q, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, const float *k_scale,
                               const float *v_scale, const int32_t *block_tables,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, float scale,
                               int max_blocks_per_seq, int num_blocks, int q_len, pa_dtype dtype,
                               int num_splits, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * pa_device_error -- synchronise `stream`, then return PA_OK or the first error
 * recorded by a kernel on the current device since the last clear
 * (PA_ERR_DEVICE_TIMEOUT takes precedence over PA_ERR_DEVICE_CHECK).  With
 * clear != 0 the word is reset to zero.  Returns PA_ERR_CUDA if the
 * synchronisation itself fails.
 */
PA_API pa_status pa_device_error(void *stream, int clear);

/*
 * pa_selftest_wait_timeout -- diagnostic: launches one thread that waits, with the
 * same bounded wait the attention kernels use for their TMA stages, on a
 * shared-memory barrier that nothing ever completes.  After about two seconds the
 * wait gives up and records PA_ERR_DEVICE_TIMEOUT in the device error word
 * (read it with pa_device_error); the CUDA context stays usable.  Lets a caller
 * check the failure path without faulting or hanging the GPU.
 */
PA_API pa_status pa_selftest_wait_timeout(void *stream);

/*
 * pa_decode_split_noalloc -- the split-KV pair (pa_decode_partial, then
 * pa_decode_combine) with its workspace in a fixed device array that the library
 * owns, for callers that cannot allocate device memory where they run attention:
 * a plug-in whose host runtime owns every device allocation, or a serving loop
 * that must not allocate (nor risk the implicit device synchronisation of
 * cudaMalloc/cudaFree) once it is running.  The pages have no counterpart; this
 * is an allocation-free convenience of this library, not a step of the method.
 *
 * Arguments are those of pa_decode_partial without the workspace; out is written
 * as by pa_decode_combine.  The array holds PA_NOALLOC_SCRATCH_BYTES on every
 * device that loads the library, until the process exits.  If
 * pa_decode_workspace_size(num_seqs, num_q_heads, q_len, head_dim, num_splits)
 * exceeds it, the call returns PA_ERR_INVALID_ARG and launches nothing.  No
 * device memory is allocated or freed.  All calls on a device share the array:
 * calls that can overlap on the GPU (unordered streams) race.  The first call on
 * a device looks up the array's device address with that device current; make
 * it before any stream capture.  The address is kept for the life of the
 * process: do not use the library across a cudaDeviceReset of that device (the
 * same holds for the error word of pa_device_error).
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
PA_API pa_status pa_decode_split_noalloc(void *out, const void *q, const void *k_cache,
                                         const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, float scale, int num_splits,
                                         int max_blocks_per_seq, int num_blocks, int q_len,
                                         pa_dtype dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
