// pa_api.cpp -- the C ABI of libpa.so: argument validation and dispatch.
// Every entry point is declared, with its contract, in include/pa.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

thread_local int t_last_launches = 0;
thread_local int t_last_partition = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_head_dim(int d) { return d == 64 || d == 128; }

// Head counts above this are refused: row and block byte counts stay far inside int.
constexpr int kMaxHeads = 1 << 16;

int check_decode(const void* out, const void* query, const void* key_cache, const void* value_cache,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                 int64_t num_blocks, int max_context_len, float scale, int dtype, int partition) {
    if (num_seqs < 0 || q_len < 1 || num_heads < 1 || num_kv_heads < 1 || max_blocks_per_seq < 1 ||
        num_blocks < 1 || max_context_len < 1)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (partition < 0 || partition % PA_BLOCK_SIZE != 0) return PA_ERR_INVALID_ARG;
    if (block_size != PA_BLOCK_SIZE || !supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
    if (num_heads > kMaxHeads) return PA_ERR_UNSUPPORTED;
    if ((int64_t)(num_heads / num_kv_heads) * q_len > 65536) return PA_ERR_UNSUPPORTED;
    if ((int64_t)max_context_len > (int64_t)max_blocks_per_seq * PA_BLOCK_SIZE) return PA_ERR_INVALID_ARG;
    if (num_blocks > (int64_t)INT32_MAX) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_tables) & 3u) != 0) return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(context_lens) & 3u) != 0) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa::DecodeArgs decode_args(void* out, const void* query, const void* key_cache, const void* value_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int64_t num_blocks, int max_context_len, float scale, int dtype, int partition_size,
                           void* workspace) {
    pa::DecodeArgs a;
    a.out = out;
    a.query = query;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.q_len = q_len;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.max_context_len = max_context_len;
    a.scale = scale;
    a.dtype = dtype;
    a.partition = partition_size == 0 ? PA_DEFAULT_PARTITION : partition_size;
    a.partition_auto = partition_size == 0;
    a.workspace = workspace;
    return a;
}

int run_decode(const pa::DecodeArgs& a, void* stream) {
    int launches = 0, part = 0;
    const int rc = pa::launch_decode(a, static_cast<cudaStream_t>(stream), &launches, &part);
    t_last_launches = launches;
    t_last_partition = part;
    return rc;
}

}  // namespace

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown status";
    }
}

int pa_last_launch_count(void) { return t_last_launches; }

int pa_last_partition_size(void) { return t_last_partition; }

int pa_reshape_and_cache(const void* key, const void* value, void* key_cache, void* value_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int dtype, void* stream) {
    t_last_launches = 0;
    if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1) return PA_ERR_INVALID_ARG;
    if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_INVALID_ARG;
    if (block_size != PA_BLOCK_SIZE || !supported_head_dim(head_dim) || num_kv_heads > kMaxHeads)
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    const int row_bytes = num_kv_heads * head_dim * 2;
    int launches = 0;
    const int st = pa::launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, num_tokens,
                                                row_bytes, num_blocks * block_size,
                                                static_cast<cudaStream_t>(stream), &launches);
    t_last_launches = launches;
    return st;
}

int pa_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping, int64_t num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int dtype, void* stream) {
    t_last_launches = 0;
    if (num_pairs < 0 || num_kv_heads < 1 || num_blocks < 1) return PA_ERR_INVALID_ARG;
    if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_INVALID_ARG;
    if (block_size != PA_BLOCK_SIZE || !supported_head_dim(head_dim) || num_kv_heads > kMaxHeads)
        return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!key_cache || !value_cache || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key_cache) || !aligned16(value_cache) || (reinterpret_cast<uintptr_t>(block_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    int launches = 0;
    const int st = pa::launch_copy_blocks(key_cache, value_cache, block_mapping, num_pairs,
                                          block_size * num_kv_heads * head_dim * 2, num_blocks,
                                          static_cast<cudaStream_t>(stream), &launches);
    t_last_launches = launches;
    return st;
}

int pa_spec_verify(int32_t* num_accepted, int32_t* out_tokens, const float* target_probs, const float* draft_probs,
                   const int32_t* draft_tokens, const float* u_accept, const float* u_sample, int num_seqs,
                   int num_draft, int vocab, void* stream) {
    t_last_launches = 0;
    if (num_seqs < 0 || num_draft < 0 || num_draft > 64 || vocab < 1) return PA_ERR_INVALID_ARG;
    if (vocab > 262144) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!num_accepted || !out_tokens || !target_probs || !u_sample) return PA_ERR_INVALID_ARG;
    if (num_draft > 0 && (!draft_probs || !draft_tokens || !u_accept)) return PA_ERR_INVALID_ARG;
    const void* ptrs[] = {num_accepted, out_tokens, target_probs, draft_probs, draft_tokens, u_accept, u_sample};
    for (const void* q : ptrs)
        if ((reinterpret_cast<uintptr_t>(q) & 3u) != 0) return PA_ERR_INVALID_ARG;
    int launches = 0;
    const int st = pa::launch_spec_verify(num_accepted, out_tokens, target_probs, draft_probs, draft_tokens, u_accept,
                                          u_sample, num_seqs, num_draft, vocab, static_cast<cudaStream_t>(stream),
                                          &launches);
    t_last_launches = launches;
    return st;
}

size_t pa_decode_workspace_size_ex(int num_seqs, int q_len, int num_heads, int head_dim, int max_context_len,
                                   int partition_size) {
    if (num_seqs < 0 || q_len < 1 || num_heads < 1 || head_dim < 1 || max_context_len < 1) return 0;
    if (partition_size == 0) partition_size = PA_DEFAULT_PARTITION;
    if (partition_size < 0 || partition_size % PA_BLOCK_SIZE != 0) return 0;
    return pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, partition_size).total;
}

size_t pa_decode_workspace_size(int num_seqs, int q_len, int num_heads, int head_dim, int max_context_len) {
    return pa_decode_workspace_size_ex(num_seqs, q_len, num_heads, head_dim, max_context_len, 0);
}

int pa_decode_attention_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                           const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, int max_context_len, float scale, int dtype,
                           int partition_size, void* workspace, size_t workspace_bytes, void* stream) {
    t_last_launches = 0;
    const int st = check_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, max_context_len, scale, dtype, partition_size);
    if (st != PA_OK || num_seqs == 0) return st;
    const pa::DecodeArgs a = decode_args(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                         context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim,
                                         num_blocks, max_context_len, scale, dtype, partition_size, workspace);
    const size_t need = pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, a.partition).total;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    return run_decode(a, stream);
}

int pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache, void* value_cache,
                             const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads, int head_dim,
                             int block_size, int64_t num_blocks, int dtype, float k_scale, float v_scale,
                             void* stream) {
    t_last_launches = 0;
    if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1) return PA_ERR_INVALID_ARG;
    if (dtype != PA_BF16 && dtype != PA_FP16) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (block_size != PA_BLOCK_SIZE || !supported_head_dim(head_dim) || num_kv_heads > kMaxHeads)
        return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
        return PA_ERR_INVALID_ARG;
    int launches = 0;
    const int st = pa::launch_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, num_tokens,
                                                    num_kv_heads * head_dim, num_blocks * block_size, dtype, k_scale,
                                                    v_scale, static_cast<cudaStream_t>(stream), &launches);
    t_last_launches = launches;
    return st;
}

int pa_decode_attention_fp8kv(void* out, const void* query, const void* key_cache, const void* value_cache,
                              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                              int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim, int block_size,
                              int64_t num_blocks, int max_context_len, float scale, int dtype, float k_scale,
                              float v_scale, int partition_size, void* workspace, size_t workspace_bytes,
                              void* stream) {
    t_last_launches = 0;
    const int st = check_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, max_context_len, scale, dtype, partition_size);
    if (st != PA_OK || num_seqs == 0) return st;
    if (head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || !(k_scale > 0.f) || !(v_scale > 0.f))
        return PA_ERR_INVALID_ARG;
    pa::DecodeArgs a = decode_args(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, num_blocks,
                                   max_context_len, scale, dtype, partition_size, workspace);
    const size_t need = pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, a.partition).total;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    a.fp8 = true;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return run_decode(a, stream);
}

int pa_decode_attention(void* out, const void* query, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        int64_t num_blocks, int max_context_len, float scale, int dtype, void* workspace,
                        size_t workspace_bytes, void* stream) {
    return pa_decode_attention_ex(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, 1, num_heads, num_kv_heads, head_dim, block_size,
                                  num_blocks, max_context_len, scale, dtype, 0, workspace, workspace_bytes, stream);
}

int pa_decode_attention_multiquery(void* out, const void* query, const void* key_cache, const void* value_cache,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int q_len, int num_heads,
                                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                   int max_context_len, float scale, int dtype, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    return pa_decode_attention_ex(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                  context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                  num_blocks, max_context_len, scale, dtype, 0, workspace, workspace_bytes, stream);
}

int pa_decode_attention_noalloc(void* out, const void* query, const void* key_cache, const void* value_cache,
                                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                int num_seqs, int q_len, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int64_t num_blocks, int max_context_len, float scale, int dtype,
                                int partition_size, void* stream) {
    t_last_launches = 0;
    const int st = check_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, max_context_len, scale, dtype, partition_size);
    if (st != PA_OK || num_seqs == 0) return st;
    pa::DecodeArgs a = decode_args(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, num_blocks,
                                   max_context_len, scale, dtype, partition_size, nullptr);
    // A call the tcgen05 kernel runs (no split) needs no scratch at all.
    if (pa::use_prefill_tc(a)) return run_decode(a, stream);
    const size_t need = pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, a.partition).total;
    if (need > (size_t)PA_NOALLOC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;  // too big for the fixed scratch
    if (const int ws = pa::noalloc_workspace(&a.workspace)) return ws;
    return run_decode(a, stream);
}

size_t pa_decode_workspace_size_shared_prefix(int num_seqs, int q_len, int num_heads, int head_dim,
                                              int max_context_len, int partition_size) {
    if (num_seqs < 0 || q_len < 1 || num_heads < 1 || head_dim < 1 || max_context_len < 1) return 0;
    if (partition_size == 0) partition_size = pa::kMinPrefixPartition;
    if (partition_size < 0 || partition_size % PA_BLOCK_SIZE != 0) return 0;
    return pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, partition_size, true).total;
}

int pa_decode_attention_shared_prefix(void* out, const void* query, const void* key_cache, const void* value_cache,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      const int32_t* context_lens, int num_seqs, int q_len, int num_heads,
                                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                      int max_context_len, float scale, int dtype, int num_groups,
                                      const int32_t* group_seq_start, const int32_t* group_prefix_len,
                                      int partition_size, void* workspace, size_t workspace_bytes, void* stream) {
    t_last_launches = 0;
    const int st = check_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, block_size,
                                num_blocks, max_context_len, scale, dtype, partition_size);
    if (st != PA_OK) return st;
    if (num_groups < 0 || num_groups > PA_MAX_PREFIX_GROUPS) return PA_ERR_INVALID_ARG;
    if (num_groups > 0 && (!group_seq_start || !group_prefix_len)) return PA_ERR_INVALID_ARG;
    // The group table, validated on the host and handed to the kernels by value.
    pa::PrefixGroups g;
    g.n = num_groups;
    g.tile_start[0] = 0;
    g.seq_start[0] = 0;
    const int group = num_heads / num_kv_heads;
    for (int k = 0; k <= num_groups && num_groups > 0; ++k) {
        const int v = group_seq_start[k];
        if (v < 0 || v > num_seqs || (k > 0 && v < g.seq_start[k - 1])) return PA_ERR_INVALID_ARG;
        g.seq_start[k] = v;
    }
    for (int k = 0; k < num_groups; ++k) {
        const int len = group_prefix_len[k];
        if (len < 0 || len % PA_BLOCK_SIZE != 0 || (len > 0 && len > max_context_len - q_len))
            return PA_ERR_INVALID_ARG;
        g.len[k] = len;
        const long long rows = (long long)(g.seq_start[k + 1] - g.seq_start[k]) * group * q_len;
        const long long tiles = len > 0 ? (long long)num_kv_heads * ((rows + 127) / 128) : 0;
        const long long next = g.tile_start[k] + tiles;
        if (next > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
        g.tile_start[k + 1] = (int)next;
    }
    if (num_seqs == 0) return PA_OK;
    pa::DecodeArgs a = decode_args(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   context_lens, num_seqs, q_len, num_heads, num_kv_heads, head_dim, num_blocks,
                                   max_context_len, scale, dtype, partition_size, workspace);
    if (partition_size == 0) a.partition = pa::kMinPrefixPartition;
    const size_t need =
        pa::ws_layout(num_seqs, q_len, num_heads, head_dim, max_context_len, a.partition, true).total;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    a.groups = &g;
    return run_decode(a, stream);
}

int pa_get_device_error(int32_t* host_flags, int clear, void* stream) {
    if (!host_flags) return PA_ERR_INVALID_ARG;
    return pa::read_device_error(host_flags, clear, static_cast<cudaStream_t>(stream));
}

int pa_set_decode_math(int math) { return pa::set_decode_math(math); }

int pa_profile_enable(int on) { return pa::profile_enable(on); }

int pa_profile_read(float* total_ms, int* launches) {
    if (!total_ms || !launches) return PA_ERR_INVALID_ARG;
    float plan = 0.f, merge = 0.f;
    return pa::profile_read_parts(&plan, total_ms, &merge, launches);
}

int pa_profile_read_parts(float* plan_ms, float* main_ms, float* merge_ms, int* calls) {
    if (!plan_ms || !main_ms || !merge_ms || !calls) return PA_ERR_INVALID_ARG;
    return pa::profile_read_parts(plan_ms, main_ms, merge_ms, calls);
}

int pa_set_wait_limit_ns(unsigned long long ns) { return pa::set_wait_limit_ns(ns); }

}  // extern "C"
