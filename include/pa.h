/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV decode-attention library (libpa.so).
 *
 * The library implements one decode step's hot path of a PagedAttention-style
 * serving engine:
 *   1. the KV append ("reshape and cache"): the newest positions' K/V rows are
 *      written into their slots of the paged pool;
 *   2. decode attention: every sequence's query rows attend over the K/V of all
 *      its positions, which live in fixed 16-token blocks scattered through the
 *      pool and are found through the sequence's block table.
 *
 * Sources (three web pages; cited by title and section):
 *   [P1] "每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速", section
 *        "KV Cache 又大又碎，为何不用操作系统分页的思路管它？": fixed-size blocks in
 *        one pool, the block table (logical -> physical block), block size 16,
 *        blockwise attention s_j = q^T K_j / sqrt(d_k), o = sum_j softmax(s)_j V_j,
 *        equal to attention over the blocks concatenated in logical order;
 *        read-only sharing of one physical block by several sequences.
 *   [P2] "现代 LLM 推理引擎剖析", section 1.3 (KV cache manager, block layout
 *        2 x block_size x num_kv_heads x head_size x dtype bytes per layer) and
 *        section 1.6 (prepare inputs builds the slot mapping; forward runs the
 *        paged attention kernel).
 *   [P3] "LLM 推理优化的系统视角", section 3.1 (dense causal attention
 *        O_t = softmax(Q_t K_{1:t}^T / sqrt(d_h)) V_{1:t}; a decode step reads the
 *        cache and appends the new position's K/V) and section 3.2 (MHA / MQA /
 *        GQA: groups of query heads share one K/V head).
 *   Speculative verification of gamma draft tokens plus one (P1, section
 *   "对症下药": the large model checks gamma + 1 positions in one forward) is the
 *   multi-query entry point below.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, owned by the caller, C-contiguous,
 *     16-byte aligned.  The library never allocates device memory, never frees
 *     caller memory and never synchronises the stream (pa_get_device_error,
 *     pa_profile_read and pa_profile_read_parts are the documented
 *     exceptions: they wait for the stream or the recorded events).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the
 *     legacy default stream) of the current device.
 *   - 16-bit element types: PA_BF16 (bfloat16) or PA_FP16 (IEEE binary16).
 *     Arithmetic is fp32 inside the kernels; outputs are rounded once (round to
 *     nearest even) to the input type.
 *   - Pool layout: key_cache and value_cache are separate tensors, each
 *     [num_blocks, block_size, num_kv_heads, head_dim] with head_dim fastest.
 *     Token p of sequence i is at block block_tables[i][p / 16], offset p % 16.
 *   - Query head h uses kv head h / (num_heads / num_kv_heads).
 *   - context_lens[i] counts every position of sequence i INCLUDING the q_len
 *     positions being decoded (their K/V must already be appended).
 *   - Supported: head_dim 64 or 128; block_size 16;
 *     (num_heads / num_kv_heads) * q_len <= 65536.
 *   - Host-side argument errors return a status and enqueue nothing.  Device
 *     contents (block ids, lengths, slots) are checked inside the kernels: a
 *     bad value sets a bit in the library's device error word (see
 *     pa_get_device_error) and the offending read or write is skipped; the
 *     kernels never trap.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_BF16 = 0, PA_FP16 = 1 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, inconsistent sizes */
    PA_ERR_UNSUPPORTED = 2,   /* head_dim, block_size, group x q_len or a head count (> 65536) outside what is compiled */
    PA_ERR_WORKSPACE = 3,     /* workspace missing or smaller than pa_decode_workspace_size() */
    PA_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} pa_status;

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID 0x1  /* a block-table entry in use lies outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT  0x2  /* context_lens[i] < q_len, < 1, > max_context_len or beyond the table */
#define PA_DEVERR_SLOT     0x4  /* slot_mapping[t] >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT  0x8  /* a bounded wait inside a kernel gave up (internal error) */
#define PA_DEVERR_INTERNAL 0x10 /* a kernel refused an inconsistent launch configuration (library bug) */
#define PA_DEVERR_TOKEN    0x20 /* a draft token outside [0, vocab) (treated as rejected) */
#define PA_DEVERR_QUERY_RANGE 0x40 /* FP8 caches: a bf16 query element of magnitude >= 65520 (beyond fp16) */

#define PA_BLOCK_SIZE 16
#define PA_DEFAULT_PARTITION 512  /* tokens per split-K partition */

/*
 * KV append ([P3] section 3.1, decode-step state change; slot mapping from [P2]
 * section 1.6).  For every new token t with slot = slot_mapping[t] >= 0:
 *   key_cache  [slot / block_size, slot % block_size, :, :] = key  [t, :, :]
 *   value_cache[slot / block_size, slot % block_size, :, :] = value[t, :, :]
 * a byte-exact copy.  Negative slots are padding and write nothing; slots
 * >= num_blocks * block_size set PA_DEVERR_SLOT and write nothing.
 *   key, value   [num_tokens, num_kv_heads, head_dim], read
 *   key_cache,   [num_blocks, block_size, num_kv_heads, head_dim], written
 *   value_cache
 *   slot_mapping [num_tokens] int64, read
 * num_tokens == 0 is a no-op.
 */
int pa_reshape_and_cache(const void* key, const void* value, void* key_cache, void* value_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, int dtype, void* stream);

/*
 * Copy-on-write block copy ([P1] section on paged KV: blocks shared by several
 * sequences carry a reference count; a sequence about to write into a shared
 * block first gets its own copy, and only that one block is copied).  For every
 * pair i of block_mapping [num_pairs, 2] int64 = (src, dst):
 *   key_cache[dst] = key_cache[src], value_cache[dst] = value_cache[src]
 * whole [block_size, num_kv_heads, head_dim] blocks, byte for byte.
 * Contract: the dst blocks are distinct and none is also a src of the same call
 * (the caller's block manager copies into freshly allocated blocks); otherwise
 * the result depends on copy order.  Pairs with an id outside [0, num_blocks)
 * set PA_DEVERR_BLOCK_ID and copy nothing.  num_pairs == 0 is a no-op.
 * The table update (and the following pa_reshape_and_cache) are the caller's.
 */
int pa_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping, int64_t num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int dtype,
                   void* stream);

/*
 * Speculative-decoding verification ([P2] section 2.4 Speculative Decoding, steps
 * 3-4; [P1] section "对症下药" on checking gamma + 1 positions in one forward).
 * Per sequence n, with k = num_draft draft tokens:
 *   scan i = 0 .. k-1: t = draft_tokens[n][i];
 *     accept if p_large[i][t] >= p_draft[i][t], else accept if
 *     u_accept[n][i] < p_large[i][t] / p_draft[i][t] (IEEE fp32 division);
 *     at the first rejection stop and draw a token from (p_large[i] - p_draft[i])+
 *     (from p_large[i] if that residual is all zero);
 *   if all k drafts are accepted, draw the bonus token from p_large[k].
 * A draw with uniform u over weights w takes the smallest v whose prefix sum of
 * w exceeds u times the total, computed on w converted exactly to 2^-40 fixed
 * point and u to 2^-24 (integer-exact, order independent).
 *   num_accepted [N] int32, written: accepted drafts, 0..k
 *   out_tokens   [N, k+1] int32, written: accepted drafts, the drawn token, then -1
 *   target_probs [N, k+1, V] fp32; draft_probs [N, k, V] fp32; draft_tokens [N, k]
 *   int32; u_accept [N, k] fp32 in [0,1); u_sample [N] fp32 in [0,1) (the caller
 *   draws the random numbers).
 * 0 <= num_draft <= 64; V <= 262,144.  A draft token outside [0, V) sets PA_DEVERR_TOKEN and
 * counts as a rejection.
 */
int pa_spec_verify(int32_t* num_accepted, int32_t* out_tokens, const float* target_probs,
                   const float* draft_probs, const int32_t* draft_tokens, const float* u_accept,
                   const float* u_sample, int num_seqs, int num_draft, int vocab, void* stream);

/*
 * Bytes of device workspace pa_decode_attention* needs for these sizes and the
 * default partition (PA_DEFAULT_PARTITION tokens).  The workspace holds the
 * per-call work list and the split-K partials (fp32 m, l and unnormalised o
 * per partition); it needs no initialisation and may be reused by every call
 * on the same stream.
 */
size_t pa_decode_workspace_size(int num_seqs, int q_len, int num_heads, int head_dim,
                                int max_context_len);

/* Same, for an explicit partition size in tokens (a positive multiple of 16). */
size_t pa_decode_workspace_size_ex(int num_seqs, int q_len, int num_heads, int head_dim,
                                   int max_context_len, int partition_size);

/*
 * Paged decode attention, one query token per sequence ([P1] blockwise
 * attention; [P3] section 3.1 dense definition it equals; [P3] section 3.2
 * GQA).  For sequence i, query head h, kv head g = h / (num_heads/num_kv_heads),
 * L = context_lens[i]:
 *   out[i, h, :] = sum_p softmax_p(scale * q[i, h, :] . K_i[p, g, :]) V_i[p, g, :],
 *   p = 0 .. L-1,
 * where K_i / V_i are the sequence's blocks in logical order.
 *   out          [num_seqs, num_heads, head_dim], written
 *   query        [num_seqs, num_heads, head_dim], read
 *   key_cache,   [num_blocks, 16, num_kv_heads, head_dim], read
 *   value_cache
 *   block_tables [num_seqs, max_blocks_per_seq] int32, read; entries past
 *                ceil(L/16) are never read
 *   context_lens [num_seqs] int32, read; each in [1, max_context_len]
 *   max_context_len  an upper bound of every context_lens[i] (sizes the workspace)
 *   workspace    device scratch of at least pa_decode_workspace_size() bytes
 * Sequences longer than one partition are split into partitions (512-2048 tokens,
 * chosen by the library; see pa_decode_attention_ex) whose fp32 partial results are
 * merged by their log-sum-exp.
 * Sequences with invalid lengths leave their output rows unwritten and set
 * PA_DEVERR_CONTEXT.
 */
int pa_decode_attention(void* out, const void* query, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                        int head_dim, int block_size, int64_t num_blocks, int max_context_len,
                        float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Multi-query decode attention: q_len query rows per sequence (gamma draft
 * tokens + 1 for speculative verification, or a prefill chunk), causal inside
 * the chunk.  Row j of sequence i is position L - q_len + j and attends
 * positions 0 .. L - q_len + j.
 *   out, query [num_seqs, q_len, num_heads, head_dim]
 * Everything else as pa_decode_attention; each context_lens[i] must be >= q_len.
 *
 * Prefill chunks ("现代 LLM 推理引擎剖析", section 2.1 Chunked Prefill: a long
 * prompt runs in chunks, each attending to the cache its earlier chunks
 * filled) are this same call with q_len = the chunk length.  When a kv head has
 * at least 128 query rows (num_heads / num_kv_heads * q_len) and the library
 * chooses the split (partition size 0), the call runs as one tcgen05 kernel:
 * 128-row query tiles, S and O accumulated in tensor memory, the softmax weights
 * rounded once to the input type for the P.V product, no split of the context.
 * The workspace is then not used.
 */
int pa_decode_attention_multiquery(void* out, const void* query, const void* key_cache,
                                   const void* value_cache, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                   int q_len, int num_heads, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, int max_context_len,
                                   float scale, int dtype, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * General form of the two calls above with an explicit split-K partition size
 * (tokens, a positive multiple of 16).  0 lets the library choose: 512, 1024 or
 * 2048 tokens, the largest that still leaves about three work units per resident
 * CTA when each sequence is taken as max_context_len / 2 long (fewer partials to
 * merge, the hand-out still balanced); pa_last_partition_size() reports it.  A
 * partition size >= max_context_len computes every sequence in one piece (no
 * merge).  The workspace must be sized with pa_decode_workspace_size_ex() for the
 * same partition size (0: PA_DEFAULT_PARTITION, which covers every choice).
 * Results agree across partition sizes within fp32 rounding.
 */
int pa_decode_attention_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int q_len, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           int max_context_len, float scale, int dtype, int partition_size,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Multi-query decode attention over sequences that share a prefix of pool blocks.
 * Where sequences share blocks ([P1] section "KV Cache 又大又碎，为何不用操作系统分页的
 * 思路管它？": parallel samples share one prompt, beam-search branches a prefix, and one
 * physical block is mapped by the logical blocks of many sequences under a reference count;
 * [P2] section 1.6 and its prefix-caching example: requests that hit the same cached prefix
 * blocks reuse them), the prefix's K/V are the same for every sharing sequence.  This call
 * computes exactly what pa_decode_attention_multiquery computes, but attends the shared
 * prefix once per kv head for the query rows of all sequences of a group together (on the
 * tcgen05 tensor cores, 128 rows at a time), the rest of each sequence with the split-K
 * partition pass, and merges the pieces by their log-sum-exp (the blockwise softmax of [P1]
 * and the tiling of [P3] section 4.2 change the order of the sums, not the result).
 *
 * Groups (HOST arrays, read before the call returns):
 *   num_groups        0 .. PA_MAX_PREFIX_GROUPS
 *   group_seq_start   [num_groups + 1], non-decreasing, in [0, num_seqs]: group k is
 *                     sequences group_seq_start[k] .. group_seq_start[k + 1] - 1; sequences
 *                     outside [group_seq_start[0], group_seq_start[num_groups]) share nothing
 *   group_prefix_len  [num_groups] positions, a multiple of 16 (whole blocks), 0 for a group
 *                     that shares nothing, and at most max_context_len - q_len
 * Contract: every sequence i of group k maps its block-table entries 0 .. len/16 - 1 to the
 * same physical blocks as the group's first sequence (only the first sequence's entries are
 * read), and context_lens[i] - q_len >= len (the chunk's rows lie after the prefix and each
 * sees all of it); a sequence that breaks the length rule sets PA_DEVERR_CONTEXT and its rows
 * are left untouched.  Everything else as pa_decode_attention_multiquery (16-bit caches; the
 * prefix pass uses the tcgen05 kernel whatever pa_set_decode_math says).  The workspace must
 * hold pa_decode_workspace_size_shared_prefix() bytes for the same partition size (0: the
 * library chooses 512 to 2048 tokens for the positions after the prefixes).  Results agree
 * with pa_decode_attention_multiquery within fp32 rounding.
 */
#define PA_MAX_PREFIX_GROUPS 256

size_t pa_decode_workspace_size_shared_prefix(int num_seqs, int q_len, int num_heads, int head_dim,
                                              int max_context_len, int partition_size);

int pa_decode_attention_shared_prefix(void* out, const void* query, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                      int q_len, int num_heads, int num_kv_heads, int head_dim,
                                      int block_size, int64_t num_blocks, int max_context_len, float scale,
                                      int dtype, int num_groups, const int32_t* group_seq_start,
                                      const int32_t* group_prefix_len, int partition_size, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Decode attention that allocates nothing, not even a workspace argument.
 * (The pages describe no such call; it exists for callers of this library.)
 *
 * Some callers cannot hand the library a workspace: a host program that reaches
 * the GPU only through this C ABI and has no device allocator of its own, or a
 * serving process whose allocator reserved nearly all device memory at start-up
 * for its KV pool and permits no further cudaMalloc (which would also
 * synchronise the whole device in the middle of a decode loop).  This variant
 * computes exactly what pa_decode_attention_ex computes, with the same arguments
 * minus the workspace, and takes its split-K scratch from a fixed array inside
 * the library:
 *   - the array holds PA_NOALLOC_WORKSPACE_BYTES (32 MiB) on every GPU that
 *     loads the library, until the process exits;
 *   - a call that splits (every call the tcgen05 kernel does not run, see
 *     pa_decode_attention_multiquery) and whose pa_decode_workspace_size_ex()
 *     exceeds that returns PA_ERR_WORKSPACE and enqueues nothing (use
 *     pa_decode_attention_ex then); a call the tcgen05 kernel runs uses no
 *     scratch and has no such limit;
 *   - the first call on each device looks up the array's device address (a
 *     runtime symbol query, no allocation) with that device current, and keeps
 *     it; make that first call before any stream capture.  The address belongs
 *     to the device's primary context: after cudaDeviceReset (or anything else
 *     that destroys that context) the process must not call this library on
 *     that device again, as its cached addresses (this array, the error word)
 *     and kernel attributes then refer to the old context;
 *   - every call on a device shares the one array, which keeps the last call's
 *     contents (each call rewrites all of it that it reads, so nothing needs
 *     clearing); calls that overlap on the GPU, on different streams or from
 *     different threads, race on it and must be serialised by the caller.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define PA_NOALLOC_WORKSPACE_BYTES (32u << 20)

int pa_decode_attention_noalloc(void* out, const void* query, const void* key_cache,
                                const void* value_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, int max_context_len, float scale, int dtype,
                                int partition_size, void* stream);

/*
 * FP8 KV cache ([P3] section 4.1: quantising the KV cache cuts its bytes; the
 * pages fix no format).  Caches hold one FP8 E4M3 byte per element (OCP E4M3: bias
 * 7, 3 mantissa bits, largest finite 448, no infinities), in the same
 * [num_blocks, 16, num_kv_heads, head_dim] layout, with one fp32 scale per cache
 * tensor: stored = e4m3(x / scale), read back as e4m3 * scale.
 *
 * pa_reshape_and_cache_fp8: as pa_reshape_and_cache, but key/value (16-bit, dtype)
 * are divided by k_scale / v_scale in fp32 (round to nearest) and stored as E4M3,
 * rounded to nearest even and saturated to +-448.  key_cache/value_cache are
 * uint8 [num_blocks, 16, num_kv_heads, head_dim].  Scales must be finite and > 0.
 *
 * pa_decode_attention_fp8kv: as pa_decode_attention_ex over FP8 caches (query and
 * out stay 16-bit, of dtype).  K and V bytes are widened exactly to fp16 in
 * registers; the score and P.V products run on the tensor cores in fp16 with fp32
 * accumulation (the softmax weights P rounded to fp16), k_scale folds into the
 * softmax scale and v_scale into the output.  A bf16 query is rounded to fp16 for
 * the score products: exact for elements of magnitude 2^-17 .. 65504 (smaller ones
 * are rounded to fp16's subnormal step, 2^-24).  An element of magnitude 65520 or
 * more has no fp16 value: the call still completes and raises
 * PA_DEVERR_QUERY_RANGE; the output row of that query row is undefined, the other
 * rows are unaffected.  head_dim 128 only; the workspace is sized as for
 * pa_decode_attention_ex.
 */
int pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache, void* value_cache,
                             const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads, int head_dim,
                             int block_size, int64_t num_blocks, int dtype, float k_scale, float v_scale,
                             void* stream);

int pa_decode_attention_fp8kv(void* out, const void* query, const void* key_cache, const void* value_cache,
                              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                              int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, int max_context_len, float scale, int dtype, float k_scale,
                              float v_scale, int partition_size, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Static description of a status code (never NULL). */
const char* pa_status_string(int status);

/*
 * Reads (and, if clear != 0, resets) the current device's error word after
 * waiting for `stream`.  *host_flags receives an OR of PA_DEVERR_* bits.
 */
int pa_get_device_error(int32_t* host_flags, int clear, void* stream);

/*
 * Arithmetic of the decode partition kernel, process-wide:
 *   0 (default, auto): CUDA-core fp32 FMA dot products with warp-shuffle
 *      reductions when each kv head has one query row (MHA, single token);
 *      tensor-core tiles (mma.sync m16n8k16, fp32 accumulation) for grouped
 *      heads and multi-query chunks, where they stream faster;
 *      with 128 or more query rows per kv head and the default partition, the
 *      tcgen05 prefill kernel (see pa_decode_attention_multiquery);
 *   1: CUDA-core FMA wherever a kv head has at most 8 query rows;
 *   2: mma.sync tensor-core tiles everywhere;
 *   3: the tcgen05 prefill kernel for every call over 16-bit caches, whatever
 *      the row count and partition size (FP8 caches keep their own path).
 * All agree with the fp64 definition within the output type's rounding plus
 * fp32 accumulation (the tcgen05 kernel also rounds P once).  Returns
 * PA_ERR_INVALID_ARG for other values.  Not thread safe: set it before
 * launching work.
 */
int pa_set_decode_math(int math);

/*
 * Timing hook for benchmarks.  pa_profile_enable(1) makes every following
 * decode call record CUDA events on the call's stream around its kernels (up to
 * 2048 calls): before the plan kernel, before the main kernel (the split-K
 * partition pass, or the tcgen05 kernel), after it, and after the merge kernel.
 * pa_profile_enable(2) records the same marks except the one between the main
 * and the merge kernel, so those two keep their programmatic overlap and the
 * main figure covers both.  pa_profile_read_parts() waits for the recorded
 * events and returns the summed milliseconds of the plan, main and merge
 * kernels (merge 0 in mode 2) and the number of calls, and clears the record;
 * pa_profile_read() returns the main figure only (and clears the record too).
 * pa_profile_enable(0) stops recording; changing the mode clears the record.
 * Events between kernels suspend their programmatic overlap, so a recorded
 * call runs a little slower than an unrecorded one.
 */
int pa_profile_enable(int on);
int pa_profile_read(float* total_ms, int* launches);
int pa_profile_read_parts(float* plan_ms, float* main_ms, float* merge_ms, int* calls);

/*
 * Limit of the kernels' pipeline waits (a test hook for their failure path:
 * every mbarrier wait inside a kernel gives up after a limit, sets
 * PA_DEVERR_TIMEOUT and stops the CTA, and the context stays usable).  Launches made after this
 * call use `ns` nanoseconds; 0 restores the default (2 s).  A limit below the
 * default also makes those waits poll without suspending, so a test can make
 * them run out on an ordinary call.  The waits a CTA makes for its own copies
 * and tensor-core products before it exits keep the default limit, so no CTA
 * leaves work in flight.  Process-wide; not thread safe.
 */
int pa_set_wait_limit_ns(unsigned long long ns);

/*
 * Split-K partition (tokens) the last decode call on this thread used: the caller's size,
 * the library's choice when it passed 0, or 0 when the tcgen05 kernel ran without splitting.
 */
int pa_last_partition_size(void);

/* Number of kernel launches the last decode call on this thread enqueued. */
int pa_last_launch_count(void);

/* Library ABI version (major * 100 + minor). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
