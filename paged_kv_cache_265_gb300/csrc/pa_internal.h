// pa_internal.h -- host-side contract between the C ABI (pa_api.cpp) and the
// kernel launchers (pa_kernels.cu).  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace pa {

// Workspace of one decode call (byte offsets from the workspace base).
//   header      int32[64]: [0] = number of work entries, [1] = dynamic work counter
//   part_start  int32[N+1]: first partial slot of each sequence (exclusive scan)
//   units       int4[N * Pmax]: work entries (sequence, first position, context length,
//               partial slot or -1), largest first
//   pml         float2[slots, q_len, Hq]: per-piece (max, sum) in log2 units
//   pacc        float[slots, q_len, Hq, D]: per-piece unnormalised outputs
// Pmax = ceil(max_context_len / partition) pieces per sequence, plus one for a shared prefix's
// piece when `prefix` (which also always reserves the partials: a grouped sequence merges its
// prefix piece with the rest even when the rest is one partition).
struct WsLayout {
    size_t header, part_start, units, pml, pacc, order, total;
    int pmax;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int num_seqs, int q_len, int num_heads, int head_dim, int max_context_len,
                          int partition, bool prefix = false) {
    WsLayout w{};
    int pmax = (max_context_len + partition - 1) / partition;
    if (pmax < 1) pmax = 1;
    if (prefix) pmax += 1;
    const size_t n = num_seqs > 0 ? (size_t)num_seqs : 0;
    const size_t slots = n * (size_t)pmax;
    size_t off = 0;
    w.header = off;
    off += 256;
    w.part_start = off;
    off += align256(4 * (n + 1));
    w.units = off;
    off += align256(16 * slots);
    w.pml = w.pacc = off;
    if (pmax > 1) {
        w.pml = off;
        off += align256(8 * slots * (size_t)q_len * (size_t)num_heads);
        w.pacc = off;
        off += align256(4 * slots * (size_t)q_len * (size_t)num_heads * (size_t)head_dim);
    }
    // Shared-prefix calls on tcgen05: the order of the suffix units (at most one per query row)
    w.order = off;
    if (prefix) off += align256(4 * n * (size_t)q_len * (size_t)num_heads);
    w.total = off;
    w.pmax = pmax;
    return w;
}

// Sequences that share a prefix of pool blocks: group k covers sequences seq_start[k] ..
// seq_start[k + 1] - 1, whose first len[k] positions (a multiple of 16; 0 = no sharing) lie in
// the same physical blocks, those named by the group's first sequence's block table.  Passed
// by value to the kernels that need it.
constexpr int kMaxPrefixGroups = 256;
struct PrefixGroups {
    int n;                                // number of groups
    int seq_start[kMaxPrefixGroups + 1];
    int len[kMaxPrefixGroups];
    int tile_start[kMaxPrefixGroups + 1]; // first prefix-kernel CTA of each group
};

// Shared-prefix positions of sequence i (0 outside every group).
__host__ __device__ inline int prefix_of(const PrefixGroups& g, int i) {
    if (g.n <= 0 || i < g.seq_start[0] || i >= g.seq_start[g.n]) return 0;
    int lo = 0, hi = g.n - 1;  // the last group whose start is <= i
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (g.seq_start[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return g.len[lo];
}

// Whether a sequence of length L can be computed: at least one position and the q_len
// query rows, within the stated bound and the block table; with a shared prefix of `skip`
// positions, every query row must see the whole prefix (L - q_len >= skip).
__host__ __device__ inline bool seq_len_valid(int L, int q_len, int skip, int max_context_len,
                                              int max_blocks_per_seq) {
    return L >= 1 && L >= q_len && L <= max_context_len && (L + 15) / 16 <= max_blocks_per_seq &&
           (skip == 0 || L - q_len >= skip);
}

struct DecodeArgs {
    void* out;
    const void* query;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int max_blocks_per_seq;
    int num_seqs;
    int q_len;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int64_t num_blocks;
    int max_context_len;
    float scale;
    int dtype;
    int partition;
    void* workspace;
    bool fp8 = false;     // key/value caches hold FP8 E4M3 bytes
    float k_scale = 1.f;  // their dequantisation scales
    float v_scale = 1.f;
    bool partition_auto = false;  // the caller passed partition size 0 (the library chooses)
    const PrefixGroups* groups = nullptr;  // shared prefixes (pa_decode_attention_shared_prefix)
};

// Launchers: return a pa_status; `launches` receives the number of kernels enqueued.
int launch_reshape_and_cache(const void* key, const void* value, void* key_cache, void* value_cache,
                             const int64_t* slot_mapping, int64_t num_tokens, int row_bytes,
                             int64_t num_slots, cudaStream_t stream, int* launches);
// `partition_used` receives the split-K partition in tokens (0: the tcgen05 kernel, no split).
int launch_decode(const DecodeArgs& a, cudaStream_t stream, int* launches, int* partition_used);
// Chunked-prefill attention on tcgen05 (pa_prefill.cu); launch_decode routes calls to it
// when use_prefill_tc() holds (that path does not split and uses no workspace).
int launch_prefill_tc(const DecodeArgs& a, cudaStream_t stream, int* launches);
bool use_prefill_tc(const DecodeArgs& a);
// The shared prefixes of a.groups on tcgen05 (pa_prefill.cu): one CTA per (group, kv head,
// 128-row tile).  Launched after the partition pass; each row's epilogue merges the prefix piece
// with the sequence's other pieces (partial slots part_start[i] + 1 ..) and writes the output.
int launch_prefix_tc(const DecodeArgs& a, const int* part_start, const float2* pml, const float* pacc,
                     cudaStream_t stream, int* launches);
// A shared-prefix call with at least kTcSuffixMinRows query rows per kv head, entirely on
// tcgen05 (pa_prefill.cu): a one-CTA kernel orders the suffix units longest first (into
// `order`), the suffix kernel (positions after each sequence's prefix; suffix pieces to partial
// slot i) takes them in that order, then the prefix kernel merges them and writes the output.
constexpr int kTcSuffixMinRows = 16;
int launch_shared_prefix_tc(const DecodeArgs& a, float2* pml, float* pacc, int* order, cudaStream_t stream,
                            int* launches);

// Smallest split-K partition the library chooses for a shared-prefix call (the workspace of a
// call with partition 0 is sized for it).
constexpr int kMinPrefixPartition = 512;
int launch_spec_verify(int32_t* num_accepted, int32_t* out_tokens, const float* target_probs,
                       const float* draft_probs, const int32_t* draft_tokens, const float* u_accept,
                       const float* u_sample, int num_seqs, int k, int vocab, cudaStream_t stream, int* launches);
int launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache, void* value_cache,
                                 const int64_t* slot_mapping, int64_t num_tokens, int row_elems, int64_t num_slots,
                                 int dtype, float k_scale, float v_scale, cudaStream_t stream, int* launches);
int launch_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping, int64_t num_pairs,
                       int block_bytes, int64_t num_blocks, cudaStream_t stream, int* launches);
int read_device_error(int32_t* flags, int clear, cudaStream_t stream);

// Device address of the library's fixed scratch array on the current device
// (looked up on the first call per device, then cached).
int noalloc_workspace(void** ptr);

// Limit (ns) of the kernels' pipeline waits for launches made from now on; 0 restores the
// default (kWaitLimitNs).  wait_limit_ns() is the current setting.
int set_wait_limit_ns(unsigned long long ns);
unsigned long long wait_limit_ns();

// Consumer arithmetic: 0 auto, 1 CUDA-core FMA, 2 mma.sync tensor-core tiles, 3 tcgen05 prefill kernel.
int set_decode_math(int math);

// Benchmark timing hook: CUDA events around each decode call's kernels.
int profile_enable(int on);
// Summed milliseconds of the plan kernel, the main kernel and the merge kernel over the
// recorded calls (waits for them), then clears the record.
int profile_read_parts(float* plan_ms, float* main_ms, float* merge_ms, int* calls);
// Inside a launcher: profile_call_begin() returns the call's record index (-1 when timing is
// off or the record is full); profile_mark(call, k, stream) records mark k (0 before the plan
// kernel, 1 before the main kernel, 2 after it, 3 after the merge) on the launch stream.
int profile_call_begin();
void profile_mark(int call, int mark, cudaStream_t stream);

// Tensor map of a 16-bit pool [num_blocks, 16, Hkv, head_dim]: one box = 64 elements of one
// kv head for the 16 positions of one block, 128-byte swizzled.
int kv_tensor_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks, int num_kv_heads,
                  int head_dim);
// Device address of the library's error word (PA_DEVERR_* bits) on the current device.
int device_error_word(int** ptr);
// Number of SMs of the current device (cached per device).
int sm_count(int* sms);
// Raises a kernel's dynamic shared-memory limit to `smem` bytes if it is lower.
int ensure_dynamic_smem(const void* fn, int smem);

// Launch with programmatic stream serialisation: the kernel may be scheduled
// before its predecessor finishes; it orders itself with griddep_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pa
