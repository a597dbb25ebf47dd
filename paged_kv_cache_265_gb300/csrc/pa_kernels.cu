// pa_kernels.cu -- sm_103a kernels of the paged-KV decode step and their launchers.
//
//   reshape_kernel  the KV append: copies each new token's [Hkv, D] K and V rows
//                   into its slot (16-byte vector copies).
//   plan_kernel     builds the work list of one decode call: (sequence,
//                   partition) entries, full partitions first, and each
//                   sequence's first partial slot.  One CTA; no host sync.
//   decode_kernel   persistent; one CTA per (sequence, partition, kv head)
//                   work unit at a time.  A producer warp streams the unit's
//                   16-token K/V blocks (found through the block table) into a
//                   ring of shared-memory stages with bulk copies completing on
//                   mbarriers; four consumer warps compute the grouped-head
//                   tile S = Q K^T and O += P V on the tensor cores
//                   (mma.sync m16n8k16, fp32 accumulate) with an online softmax,
//                   merge their partial states in shared memory and write either
//                   the final output or the partition's fp32 partial.
//   merge_kernel    merges the partitions of split sequences by log-sum-exp.
//
// The blockwise computation follows "每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM
// 推理提速", section on paged KV cache (s_j = q^T K_j / sqrt(d_k),
// o = sum_j softmax(s)_j V_j over blocks in logical order), which equals the
// dense causal attention of "LLM 推理优化的系统视角", section 3.1; the query-head
// grouping is section 3.2 of the latter.  The online softmax is the tiling idea
// named in its section 4.2 (execution order changes, semantics do not).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>
#include <utility>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// ---------------------------------------------------------------------------
// Device state owned by the library (module globals, not allocations).
// ---------------------------------------------------------------------------
__device__ int g_pa_error;                            // PA_DEVERR_* bits

constexpr int kBlock = 16;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Depth of the shared-memory ring (stages of one 16-token K+V block) and the
// number of decode CTAs meant to share an SM; the launcher picks the deepest
// ring that fits that many CTAs.
#ifndef PA_MAX_STAGES
#define PA_MAX_STAGES 8
#endif
// Query rows per work unit when a kv head has more of them than one CTA's four
// warps hold at once; and whether such units prefer 8-row warps (more resident CTAs)
// over 16-row warps.
#ifndef PA_ROW_GROUP_ROWS
#define PA_ROW_GROUP_ROWS 32
#endif
#ifndef PA_PREFER_NT1
#define PA_PREFER_NT1 1
#endif
// Query rows per kv head from which the auto mode runs a call on the tcgen05 prefill kernel.
#ifndef PA_TC_MIN_ROWS
#define PA_TC_MIN_ROWS 128
#endif
#ifndef PA_CTAS_PER_SM_NT1
#define PA_CTAS_PER_SM_NT1 4  // kernels whose warps own 8 query rows
#endif
#ifndef PA_CTAS_PER_SM_F8
// FP8-cache kernels whose warps own 8 query rows.  Same-box A/B on the GQA batch: 4 CTAs per SM
// (96 registers, 92 B of spills) 131.8 us, 5 (72 registers, 220 B) 133.0 us; with the query
// fragments read from shared memory instead (20 B of spills at 4 CTAs) 131.7 / 138.3 us.
#define PA_CTAS_PER_SM_F8 4
#endif
// Lazy running max in the tensor-core decode kernels (bit 0: FP8 caches, bit 1: 16-bit caches).
// Same-box A/B on the GQA batch (partition kernel): FP8 130.6 vs 131.9 us, 16-bit 162.7 vs 163.7 us.
#ifndef PA_LAZY_MAX
#define PA_LAZY_MAX 3
#endif
#ifndef PA_CTAS_PER_SM_NT2
#define PA_CTAS_PER_SM_NT2 2  // kernels whose warps own 16 query rows
#endif
constexpr int kMaxStages = PA_MAX_STAGES;

// ---------------------------------------------------------------------------
// KV append
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) reshape_kernel(const uint4* __restrict__ key,
                                                      const uint4* __restrict__ value,
                                                      uint4* __restrict__ key_cache,
                                                      uint4* __restrict__ value_cache,
                                                      const long long* __restrict__ slots,
                                                      long long num_tokens, int row_vecs,
                                                      long long num_slots) {
    // Launched under programmatic dependence: resident early, it touches no memory before the
    // kernel ahead of it in the stream has finished.
    griddep_launch_dependents();
    griddep_wait();
    const long long per_token = 2LL * row_vecs;
    const long long total = num_tokens * per_token;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long t = idx / per_token;
        const int rem = (int)(idx - t * per_token);
        const int which = rem >= row_vecs;  // 0 = K, 1 = V
        const int v = rem - which * row_vecs;
        const long long slot = __ldg(slots + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (rem == 0) atomicOr(&g_pa_error, PA_DEVERR_SLOT);
            continue;
        }
        const uint4* src = which ? value : key;
        uint4* dst = which ? value_cache : key_cache;
        dst[slot * row_vecs + v] = __ldg(src + t * row_vecs + v);
    }
}

// Eight 16-bit values (one 16-byte chunk) widened to fp32.
template <typename T>
__device__ __forceinline__ void unpack8(const uint4 raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (Elem<T>::kDtype == PA_BF16) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
            const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            f[2 * i] = v.x;
            f[2 * i + 1] = v.y;
        }
    }
}

// ---------------------------------------------------------------------------
// KV append into FP8 caches: each 16-bit element divided by the cache's scale in
// fp32 (round to nearest) and stored as E4M3, rounded to nearest even, saturating.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

template <typename T>
__global__ void __launch_bounds__(256) reshape_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                                          uint2* __restrict__ key_cache, uint2* __restrict__ value_cache,
                                                          const long long* __restrict__ slots, long long num_tokens,
                                                          int row_vecs, long long num_slots, float k_scale,
                                                          float v_scale) {
    griddep_launch_dependents();
    griddep_wait();  // as in reshape_kernel
    const long long per_token = 2LL * row_vecs;  // 8 elements per vector
    const long long total = num_tokens * per_token;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long t = idx / per_token;
        const int rem = (int)(idx - t * per_token);
        const int which = rem >= row_vecs;
        const int v = rem - which * row_vecs;
        const long long slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (rem == 0) atomicOr(&g_pa_error, PA_DEVERR_SLOT);
            continue;
        }
        float f[8];
        unpack8<T>(__ldg((which ? value : key) + t * row_vecs + v), f);
        const float sc = which ? v_scale : k_scale;
        uint32_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) b[i] = f32x2_to_e4m3x2(__fdiv_rn(f[2 * i], sc), __fdiv_rn(f[2 * i + 1], sc));
        (which ? value_cache : key_cache)[slot * row_vecs + v] = make_uint2(b[0] | b[1] << 16, b[2] | b[3] << 16);
    }
}

// ---------------------------------------------------------------------------
// Copy-on-write block copy: whole K and V blocks from src to dst, per pair.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ key_cache,
                                                          uint4* __restrict__ value_cache,
                                                          const long long* __restrict__ mapping,
                                                          long long num_pairs, int block_vecs,
                                                          long long num_blocks) {
    griddep_launch_dependents();
    const long long per_pair = 2LL * block_vecs;
    const long long total = num_pairs * per_pair;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long pr = idx / per_pair;
        const int rem = (int)(idx - pr * per_pair);
        const int which = rem >= block_vecs;  // 0 = K, 1 = V
        const int v = rem - which * block_vecs;
        const long long src = __ldg(mapping + 2 * pr), dst = __ldg(mapping + 2 * pr + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (rem == 0) atomicOr(&g_pa_error, PA_DEVERR_BLOCK_ID);
            continue;
        }
        uint4* base = which ? value_cache : key_cache;
        base[dst * block_vecs + v] = base[src * block_vecs + v];
    }
}

// ---------------------------------------------------------------------------
// Speculative-decoding verification ("现代 LLM 推理引擎剖析", section 2.4): accept
// drafts left to right (p_large >= p_draft, else with probability
// p_large / p_draft), then draw the correction from (p_large - p_draft)+ at the
// first rejection, or a bonus token from p_large[k] if all were accepted.
// Draws are inverse-CDF over weights converted exactly to 2^-40 fixed point, so
// prefix sums are integer-exact whatever the summation order.
//
// One cluster of kSpecCluster CTAs per sequence.  Every CTA takes the accept decisions
// (k lookups), then sums the fixed-point weights of its share of the vocabulary chunks
// (chunk j belongs to CTA j % kSpecCluster) and stores each chunk total into the shared
// memory of every CTA of the cluster; after one cluster barrier every CTA holds all totals,
// finds the threshold and the chunk holding it, and the chunk's owner scans it and writes
// the sequence's outputs.
// ---------------------------------------------------------------------------
struct SpecParams {
    int* num_accepted;
    int* out_tokens;
    const float* target;
    const float* draft;
    const int* draft_tokens;
    const float* u_accept;
    const float* u_sample;
    int k;
    int vocab;
};

#ifndef PA_SPEC_CLUSTER
#define PA_SPEC_CLUSTER 4
#endif
constexpr int kSpecCluster = PA_SPEC_CLUSTER;        // CTAs per sequence (4 or 8)
constexpr int kSpecThreads = 1024 / kSpecCluster;    // threads per CTA
constexpr int kSpecChunk = 4 * kSpecThreads;         // entries per chunk: thread t holds 4t .. 4t + 3
constexpr int kSpecMaxChunks = 262144 / kSpecChunk;  // vocabulary up to 262,144
constexpr int kSpecOwn = kSpecMaxChunks / kSpecCluster;  // chunks one CTA may own
constexpr int kSpecGroup = 8;                        // own chunks whose loads are in flight together
constexpr int kSpecStageBytes = 2 * kSpecGroup * kSpecChunk * 4;  // one group of chunks of both rows

// floor(x * 2^40) for 0 <= x < 2, built from the float's fields with integer operations (a
// float-to-64-bit conversion instruction runs at the FP64 rate): x = m * 2^(e - 150) with
// m = 1.f as a 24-bit integer (e >= 1), or x = f * 2^-149 for a subnormal (e = 0), so
// x * 2^40 = m * 2^(e - 110), an exact left shift for e >= 110, else a right shift, which
// drops exactly the fraction below 1.
__device__ __forceinline__ unsigned long long fixed40(float x) {
    const uint32_t b = __float_as_uint(x);
    const int e = (int)(b >> 23);  // x >= 0: no sign bit
    const uint32_t m = (b & 0x7fffffu) | (e ? 0x800000u : 0u);
    const int s = max(e, 1) - 110;
    return s >= 0 ? (unsigned long long)m << s : (s > -32 ? (unsigned long long)(m >> -s) : 0ull);
}

// Shared-memory staging of a group of chunks: kSpecGroup chunks of the first row, then of the
// second, filled by bulk copies that complete on `bar` (phase parity `phase`, per thread).
struct DrawStage {
    float* buf;
    uint32_t bar;
    uint32_t phase;
};

struct DrawSmem {
    unsigned long long red[kSpecThreads / 32][kSpecOwn];  // per-warp sums of this CTA's chunks
    unsigned long long tot[2][kSpecMaxChunks];            // totals of every chunk, per draw
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Stores v at this CTA's shared address `addr` in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint32_t rank, unsigned long long v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}

// Every thread of every CTA of the cluster; shared-memory stores before it (local or remote)
// are visible to every CTA after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The four weights (a - b)+ (or a) of entries v0 .. v0 + 3 (0 past the vocabulary): one 16-byte
// load per array where the rows allow it, else four scalar loads.
__device__ __forceinline__ float4 draw_weights4(const float* a, const float* b, int v0, int vocab, bool vec) {
    float4 w;
    if (vec && v0 + 3 < vocab) {
        const float4 x = __ldg(reinterpret_cast<const float4*>(a + v0));
        if (b) {
            const float4 y = __ldg(reinterpret_cast<const float4*>(b + v0));
            w = make_float4(x.x - y.x, x.y - y.y, x.z - y.z, x.w - y.w);
        } else {
            w = x;
        }
    } else {
        float e[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int v = v0 + c;
            e[c] = v < vocab ? (b ? __ldg(a + v) - __ldg(b + v) : __ldg(a + v)) : 0.f;
        }
        w = make_float4(e[0], e[1], e[2], e[3]);
    }
    w.x = w.x > 0.f ? w.x : 0.f;
    w.y = w.y > 0.f ? w.y : 0.f;
    w.z = w.z > 0.f ? w.z : 0.f;
    w.w = w.w > 0.f ? w.w : 0.f;
    return w;
}

// The four weights (a - b)+ (or a) of entries v0 .. v0 + 3 of group chunk q from the staging
// buffer (0 past the vocabulary, where the buffer holds stale values).
__device__ __forceinline__ float4 staged_weights4(const float* buf, int q, bool has_b, int v0, int vocab) {
    const float4 x = *reinterpret_cast<const float4*>(buf + q * kSpecChunk + 4 * (threadIdx.x & (kSpecThreads - 1)));
    float4 w = x;
    if (has_b) {
        const float4 y = *reinterpret_cast<const float4*>(buf + (kSpecGroup + q) * kSpecChunk + 4 * (threadIdx.x & (kSpecThreads - 1)));
        w = make_float4(x.x - y.x, x.y - y.y, x.z - y.z, x.w - y.w);
    }
    w.x = (v0 < vocab && w.x > 0.f) ? w.x : 0.f;
    w.y = (v0 + 1 < vocab && w.y > 0.f) ? w.y : 0.f;
    w.z = (v0 + 2 < vocab && w.z > 0.f) ? w.z : 0.f;
    w.w = (v0 + 3 < vocab && w.w > 0.f) ? w.w : 0.f;
    return w;
}

// Inverse-CDF draw with uniform u over weights (a - b)+ (or a), `round` (0 or 1) naming the
// draw's slot of chunk totals: the smallest v whose prefix sum of floor(w * 2^40) exceeds
// floor(floor(u * 2^24) * total / 2^24).  Returns the token in the one thread of the cluster
// that found it, -1 in every thread when all weights are 0, and -2 in the others.  Every
// thread of every CTA of the cluster must call it.
__device__ int cluster_draw(const float* a, const float* b, int vocab, float u, int round, DrawSmem& sm,
                            DrawStage& st) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t rank = cluster_rank();
    const int chunks = (vocab + kSpecChunk - 1) / kSpecChunk;
    const int own = chunks > (int)rank ? (chunks - 1 - (int)rank) / kSpecCluster + 1 : 0;
    const bool vec = ((reinterpret_cast<uintptr_t>(a) | (b ? reinterpret_cast<uintptr_t>(b) : 0)) & 15) == 0;
    // Rows 16-byte aligned with whole 16-byte chunks: each group of chunks is staged in shared
    // memory by bulk copies (one thread issues them, the bytes complete the barrier), so the
    // whole group is requested at once without a per-thread limit on loads in flight.
    const bool bulk = vec && (vocab & 3) == 0;
    // Pass 1: this CTA's chunks, kSpecGroup chunks in flight together.  The last group's
    // weights stay in registers for pass 2.
    float4 w[kSpecGroup];
    int g_last = 0;
    for (int g0 = 0; g0 < own; g0 += kSpecGroup) {
        g_last = g0;
        if (bulk) {
            __syncthreads();  // every thread is done with the buffer's previous contents
            if (t == 0) {
                fence_proxy_async_smem();
                const int ng = min(kSpecGroup, own - g0);
                uint32_t bytes = 0;
                for (int q = 0; q < ng; ++q) {
                    const int j = (g0 + q) * kSpecCluster + (int)rank;
                    bytes += 4u * (uint32_t)min(kSpecChunk, vocab - j * kSpecChunk) * (b ? 2u : 1u);
                }
                mbar_arrive_expect_tx(st.bar, bytes);
                const uint64_t pol = l2_policy_evict_first();
                for (int q = 0; q < ng; ++q) {
                    const int j = (g0 + q) * kSpecCluster + (int)rank;
                    const uint32_t nb = 4u * (uint32_t)min(kSpecChunk, vocab - j * kSpecChunk);
                    bulk_g2s(smem_addr(st.buf + q * kSpecChunk), a + (long long)j * kSpecChunk, nb, st.bar, pol);
                    if (b)
                        bulk_g2s(smem_addr(st.buf + (kSpecGroup + q) * kSpecChunk), b + (long long)j * kSpecChunk, nb,
                                 st.bar, pol);
                }
            }
            mbar_wait(st.bar, st.phase, &g_pa_error, nullptr);
            st.phase ^= 1u;
        }
#pragma unroll
        for (int q = 0; q < kSpecGroup; ++q) {
            const int v0 = ((g0 + q) * kSpecCluster + (int)rank) * kSpecChunk + 4 * t;
            w[q] = g0 + q >= own ? make_float4(0.f, 0.f, 0.f, 0.f)
                   : bulk        ? staged_weights4(st.buf, q, b != nullptr, v0, vocab)
                                 : draw_weights4(a, b, v0, vocab, vec);
        }
#pragma unroll
        for (int q = 0; q < kSpecGroup; ++q) {
            unsigned long long s = fixed40(w[q].x) + fixed40(w[q].y) + fixed40(w[q].z) + fixed40(w[q].w);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0 && g0 + q < own) sm.red[warp][g0 + q] = s;
        }
    }
    __syncthreads();
    // This CTA's chunk totals (eight warp sums each) into every CTA's table.
    for (int jl = warp; jl < own; jl += kSpecThreads / 32) {
        unsigned long long s = lane < kSpecThreads / 32 ? sm.red[lane][jl] : 0ull;
#pragma unroll
        for (int o = kSpecThreads / 64; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        s = __shfl_sync(0xffffffffu, s, 0);
        if (lane < kSpecCluster) {
            const int j = jl * kSpecCluster + (int)rank;
            st_cluster_u64(smem_addr(&sm.tot[round][j]), lane, s);
        }
    }
    cluster_sync();
    // Every warp of every CTA: prefix over all chunk totals (lane l holds chunks l * E .. + E - 1),
    // the threshold and the first chunk whose inclusive prefix exceeds it.  Every warp reaches
    // the same values from the same totals, so no barrier is needed to share them.
    constexpr int E = kSpecMaxChunks / 32;
    unsigned long long c[E];
    unsigned long long mine = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int j = lane * E + e;
        c[e] = j < chunks ? sm.tot[round][j] : 0ull;
        mine += c[e];
    }
    unsigned long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned long long total = __shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) return -1;  // every weight is 0 (every warp of every CTA agrees)
    const unsigned long long u24 = __float2ull_rz(u * 16777216.0f);
    const unsigned long long thresh = (__umul64hi(u24, total) << 40) | ((u24 * total) >> 24);
    // the lane whose range holds the first prefix above the threshold (the last lane's prefix is
    // the total, which exceeds it)
    const int l = __ffs(__ballot_sync(0xffffffffu, incl > thresh)) - 1;
    int found = -1;
    unsigned long long found_base = 0;
    if (lane == l) {
        unsigned long long run = incl - mine;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (found < 0 && run + c[e] > thresh) {
                found = lane * E + e;
                found_base = run;
            }
            run += c[e];
        }
    }
    const int chunk = __shfl_sync(0xffffffffu, found, l);
    if (chunk % kSpecCluster != (int)rank) return -2;  // another CTA owns the threshold's chunk
    // In the owner: the warp whose 4 * 32 entries of the chunk hold the threshold, from the
    // per-warp sums of pass 1.
    const int jl = chunk / kSpecCluster;
    unsigned long long before = __shfl_sync(0xffffffffu, found_base, l);
    for (int w2 = 0; w2 < warp; ++w2) before += sm.red[w2][jl];
    if (!(before <= thresh && thresh < before + sm.red[warp][jl])) return -2;
    // Pass 2, in that warp: its entries in order (each lane's four, then a warp scan), from the
    // registers of pass 1 when the chunk was in its last group.
    const int v0 = chunk * kSpecChunk + 4 * t;
    const int jg = jl - g_last;
    float4 wc;
    if (jg >= 0 && jg < kSpecGroup) {
        wc = w[0];
#pragma unroll
        for (int q = 1; q < kSpecGroup; ++q)
            if (q == jg) wc = w[q];
    } else {
        wc = draw_weights4(a, b, v0, vocab, vec);
    }
    const unsigned long long x[4] = {fixed40(wc.x), fixed40(wc.y), fixed40(wc.z), fixed40(wc.w)};
    const unsigned long long mine2 = x[0] + x[1] + x[2] + x[3];
    unsigned long long incl2 = mine2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += y;
    }
    unsigned long long run = before + (incl2 - mine2);
    int tok = -2;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (run <= thresh && run + x[q] > thresh && v0 + q < vocab) tok = v0 + q;
        run += x[q];
    }
    return tok;
}

// One cluster of kSpecCluster CTAs per sequence (grid: num_seqs * kSpecCluster).
__global__ void __launch_bounds__(kSpecThreads, kSpecCluster / 2) spec_verify_kernel(const SpecParams p) {
    griddep_launch_dependents();
    extern __shared__ __align__(128) float spec_stage[];  // kSpecStageBytes
    __shared__ __align__(8) unsigned long long s_bar;
    __shared__ DrawSmem sm;
    __shared__ int s_pos;
    __shared__ int s_ok[64];
    __shared__ int s_tokv[64];
    const int n = blockIdx.x / kSpecCluster;
    const long long V = p.vocab;
    const float* pl = p.target + (long long)n * (p.k + 1) * V;
    const float* pd = p.draft + (long long)n * p.k * V;
    int* out = p.out_tokens + (long long)n * (p.k + 1);
    // The uniforms are loaded up front, beside the draft tokens: on cold data every dependent
    // load is a DRAM round trip, and only the probability lookups depend on the tokens.
    const float u = __ldg(p.u_sample + n);
    DrawStage st{spec_stage, smem_addr(&s_bar), 0u};
    if (threadIdx.x == 0) {
        mbar_init(st.bar, 1);
        fence_barrier_init();
    }
    // Every draft position's accept decision in parallel (thread i), then the left-to-right
    // scan for the first rejection on the flags.  Every CTA of the cluster takes the same
    // decisions from the same values.
    if (threadIdx.x < p.k) {
        const int i = threadIdx.x;
        const int t = __ldg(p.draft_tokens + (long long)n * p.k + i);
        const float ua = __ldg(p.u_accept + (long long)n * p.k + i);
        bool accept = false;
        if (t < 0 || t >= p.vocab) {  // not a token: counts as a rejection
            if (cluster_rank() == 0) atomicOr(&g_pa_error, PA_DEVERR_TOKEN);
        } else {
            const float a = __ldg(pl + i * V + t), b = __ldg(pd + i * V + t);
            accept = a >= b || ua < __fdiv_rn(a, b);
        }
        s_ok[i] = accept;
        s_tokv[i] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int i = 0;
        while (i < p.k && s_ok[i]) ++i;
        s_pos = i;
    }
    __syncthreads();
    const int i = s_pos;
    int tok = cluster_draw(pl + i * V, i < p.k ? pd + i * V : nullptr, p.vocab, u, 0, sm, st);
    // An all-zero residual: the draw falls back to p_large[i] (every CTA takes this branch).
    if (tok == -1 && i < p.k) tok = cluster_draw(pl + i * V, nullptr, p.vocab, u, 1, sm, st);
    // The thread that drew the token (thread 0 of rank 0 if nothing was drawable) writes the outputs.
    if (tok >= 0 || (tok == -1 && threadIdx.x == 0 && cluster_rank() == 0)) {
        for (int jj = 0; jj < i; ++jj) out[jj] = s_tokv[jj];
        out[i] = tok;
        for (int jj = i + 1; jj <= p.k; ++jj) out[jj] = -1;
        p.num_accepted[n] = i;
    }
}

// ---------------------------------------------------------------------------
// Work list
// ---------------------------------------------------------------------------
struct PlanParams {
    const int* context_lens;
    int* header;        // [0] work entries, [1] dynamic work counter (reset here)
    int* part_start;
    int4* units;
    int num_seqs;
    int num_kv_heads;
    int q_len;
    int partition;
    int max_blocks_per_seq;
    int max_context_len;
};

// Exclusive scan of v over the 1024-thread block; `total` receives the sum.
__device__ int block_exclusive_scan(int v, int* scratch32, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch32[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = scratch32[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        scratch32[lane] = w;
    }
    __syncthreads();
    const int before = warp ? scratch32[warp - 1] : 0;
    total = scratch32[31];
    __syncthreads();
    return before + x - v;
}

// One sequence as the plan sees it: its length, the shared-prefix positions another kernel
// computes for it (0 without a prefix group), how many of its partial results the merge
// combines (`pieces`: the prefix piece, if any, then the split-K partitions of the rest;
// 0 for an invalid length, which is flagged) and its first partial slot.
struct PlanSeq {
    int len, skip, pieces, slot;
};

__device__ __forceinline__ PlanSeq plan_seq(const PlanParams& p, const PrefixGroups* g, int i) {
    PlanSeq s{0, 0, 0, 0};
    if (i >= p.num_seqs) return s;
    s.len = p.context_lens[i];
    s.skip = g ? prefix_of(*g, i) : 0;
    if (!seq_len_valid(s.len, p.q_len, s.skip, p.max_context_len, p.max_blocks_per_seq)) {
        atomicOr(&g_pa_error, PA_DEVERR_CONTEXT);
        return s;
    }
    s.pieces = (s.skip > 0) + (s.len - s.skip + p.partition - 1) / p.partition;
    return s;
}

// Size bucket of a work entry: its block count, capped; larger buckets go first.
constexpr int kPlanBuckets = 64;
__device__ __forceinline__ int part_bucket(const PlanParams& p, int L, int tok0) {
    const int nb = (min(p.partition, L - tok0) + kBlock - 1) / kBlock;
    return min(nb, kPlanBuckets - 1);
}

// One CTA: numbers each sequence's partial results (part_start), then lays the work entries
// (sequence, first position, length, partial slot or -1 when the entry is the sequence's only
// piece and writes the output itself) out largest first (a counting sort on block count), so
// that CTAs taking entries in order finish close together.  The order within a size bucket
// does not affect any result.  With prefix groups, a grouped sequence's entries cover only the
// positions after its shared prefix; its partial slot part_start[i] is the prefix piece's.
__device__ __forceinline__ void plan_body(const PlanParams& p, const PrefixGroups* g) {
    static_assert(kPlanBuckets == 64, "the bucket scan below gives each lane of one warp two buckets");
    __shared__ int scratch[32];
    __shared__ int hist[kPlanBuckets];
    if (threadIdx.x < kPlanBuckets) hist[threadIdx.x] = 0;
    __syncthreads();
    // Each thread keeps its first sequence (all of them, up to 1024 sequences) in registers
    // for the second pass.
    int carry = 0;
    PlanSeq s0{0, 0, 0, 0};
    for (int base = 0; base < p.num_seqs; base += 1024) {
        const int i = base + threadIdx.x;
        PlanSeq s = plan_seq(p, g, i);
        int tot;
        s.slot = carry + block_exclusive_scan(s.pieces, scratch, tot);
        if (i < p.num_seqs) {
            p.part_start[i] = s.slot;
            for (int tok0 = s.skip; tok0 < s.len && s.pieces > 0; tok0 += p.partition)
                atomicAdd(&hist[part_bucket(p, s.len, tok0)], 1);
        }
        if (base == 0) s0 = s;
        carry += tot;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        // Bucket starts, largest bucket first: an exclusive scan over the buckets in descending
        // order, lane l taking buckets 63 - 2l and 62 - 2l.
        const int lane = threadIdx.x;
        const int b0 = kPlanBuckets - 1 - 2 * lane, b1 = b0 - 1;
        const int n0 = hist[b0], n1 = hist[b1];
        int x = n0 + n1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const int start = x - (n0 + n1);
        hist[b0] = start;
        hist[b1] = start + n0;
        if (lane == 31) p.header[0] = x;  // work entries (every bucket counted)
        if (lane == 0) {
            p.part_start[p.num_seqs] = carry;
            p.header[1] = 0;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) {
        PlanSeq s = s0;
        if (i >= 1024) {
            s = plan_seq(p, g, i);
            s.slot = p.part_start[i];
        }
        if (s.pieces == 0) continue;
        int slot = s.pieces == 1 ? -1 : s.slot + (s.skip > 0);
        for (int tok0 = s.skip; tok0 < s.len; tok0 += p.partition) {
            const int pos = atomicAdd(&hist[part_bucket(p, s.len, tok0)], 1);
            p.units[pos] = make_int4(i, tok0, s.len, slot);
            if (slot >= 0) ++slot;
        }
    }
}

__global__ void __launch_bounds__(1024) plan_kernel(const PlanParams p) {
    griddep_launch_dependents();  // the partition pass may start its set-up now ...
    griddep_wait();               // ... but the lengths may come from the kernel before this one
    plan_body(p, nullptr);
}

__global__ void __launch_bounds__(1024) plan_prefix_kernel(const PlanParams p, const __grid_constant__ PrefixGroups g) {
    griddep_launch_dependents();
    griddep_wait();
    plan_body(p, &g);
}

// ---------------------------------------------------------------------------
// Decode attention
// ---------------------------------------------------------------------------
// K/V staging.  Each 16-token block of one kv head is fetched by tensor-map TMA
// as boxes of 16 rows x 64 elements (128 B), 128-byte swizzled in shared memory
// (16-byte chunk c of row r sits at chunk c ^ (r & 7)), so ldmatrix reads are
// bank-conflict free without padding.  A block with only `valid` < 16 tokens is
// fetched with its box starting at token coordinate valid - 16: the rows before
// coordinate 0 are outside the tensor and arrive as zeros, the tokens land in
// the last `valid` rows, and P.V never multiplies stale data.
constexpr int kBoxCols = 64;                       // elements per box row (128 B)
constexpr int kBoxBytes = kBlock * kBoxCols * 2;   // 2 KB

struct alignas(128) DecodeParams {
    CUtensorMap tmap_k;  // [num_blocks, 16, Hkv, D] viewed as 4-D, box {64, 1, 16, 1}
    CUtensorMap tmap_v;
    void* out;
    const void* query;
    const int* block_tables;
    const int* header;
    int* work_counter;   // next work unit to hand out (reset by the plan kernel)
    const int4* units;   // (seq, first position, context_len, partial slot or -1), largest first
    float2* pml;
    float* pacc;
    long long num_blocks;
    int max_blocks_per_seq;
    int q_len;
    int num_heads;
    int num_kv_heads;
    int group;         // query heads per kv head
    int rows;          // query rows per work unit: min(64, group * q_len)
    int total_rows;    // group * q_len query rows per kv head
    int row_groups;    // ceil(total_rows / rows): units per (sequence, partition, kv head)
    int partition;     // tokens per partition (multiple of 16)
    int stages;        // ring length, a multiple of block_splits, <= kMaxStages
    int mtiles;        // ceil(rows / 16) tensor-core row tiles
    int block_splits;  // kConsumerWarps / mtiles warps share a tile's blocks
    int slot_rows;     // min(8 NT, rows): rows each warp leaves in the combine buffer
    float scale_log2;  // scale * log2(e) (times the K dequantisation scale for an FP8 cache)
    float v_scale;     // V dequantisation scale (1 for 16-bit caches)
    unsigned int wait_limit_ns;  // limit of the pipeline waits (pa_set_wait_limit_ns), at most 2 s
};

// One work unit: positions tok0 .. tok0 + ntok - 1 of sequence `seq` (length len) for the kv
// head's query rows row0 .. row0 + nrows - 1; its result goes to partial slot `slot`, or
// straight to the output when slot < 0 (the sequence's only piece).
struct UnitInfo {
    int seq, tok0, len, slot, kvh, ntok, row0, nrows;
};

struct SmemLayout {
    int stage_bytes, qpitch, q_half_bytes;
    int off_q, off_comb, off_m, off_l, off_bars, off_info, off_fma, total;
};

// Offsets from a 1024-byte aligned base (the swizzled TMA boxes need that alignment).
// Per consumer warp, the CUDA-core path exchanges P (8 rows x 16 tokens) and the
// 8 rows' rescale factors through shared memory.
constexpr int kFmaWarpFloats = 8 * 16 + 8;
// Per consumer warp, slots for the running (max, sum) of up to this many query rows.
constexpr int kCombRows = 32;

__host__ __device__ inline SmemLayout smem_layout(int head_dim, int stages, int mtiles, int tile_rows, int slot_rows,
                                                  bool fma = false, bool f8 = false) {
    SmemLayout s;
    // 16-bit caches: K boxes then V boxes; FP8 caches: the K box then the V box (128 B rows); all swizzled
    s.stage_bytes = f8 ? 2 * kBlock * head_dim : 2 * (head_dim / kBoxCols) * kBoxBytes;
    s.qpitch = head_dim * 2 + 16;                            // padded query rows
    s.q_half_bytes = mtiles * tile_rows * s.qpitch;
    s.off_q = stages * s.stage_bytes;
    s.off_comb = s.off_q + 2 * s.q_half_bytes;
    s.off_m = s.off_comb + kConsumerWarps * slot_rows * head_dim * 4;
    s.off_l = s.off_m + kConsumerWarps * kCombRows * 4;
    s.off_bars = s.off_l + kConsumerWarps * kCombRows * 4;
    s.off_info = s.off_bars + (2 * kMaxStages + 4) * 8;
    s.off_fma = s.off_info + 2 * (int)sizeof(UnitInfo) + 16;
    s.total = s.off_fma + (fma ? kConsumerWarps * kFmaWarpFloats * 4 : 0) + 1024;  // + alignment slack
    return s;
}

// Byte offset of element column `col` of box row `row` inside a stage half (K or V).
__device__ __forceinline__ uint32_t swz(int row, int col) {
    const int box = col >> 6, chunk = (col & 63) >> 3;
    return box * kBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
        : "memory");
}

// Transpose of an 8x8 matrix of 16-bit values held as the standard fragment
// (lane holds row lane/4, columns 2*(lane%4) and +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// bar.red.or over the 128 consumer threads (named barrier 1): every thread
// gets the OR of `v` across them.
__device__ __forceinline__ bool consumers_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q, r;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred r, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, r;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Sum of 8 per-row partials over the 2^LCH lanes of a lane group, transposed: three
// halving exchange stages on lane bits LCH-1, LCH-2, LCH-3 leave each lane with the total
// of row ((lane >> (LCH-3)) & 7); remaining lower bits are summed as a plain all-reduce.
template <int LCH>
__device__ __forceinline__ float transpose_reduce8(const float (&part)[8], int lane) {
    constexpr int b0 = LCH - 1, b1 = LCH - 2, b2 = LCH - 3;
    float a4[4], a2[2];
    const bool h0 = (lane >> b0) & 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = h0 ? part[i] : part[i + 4];
        const float keep = h0 ? part[i + 4] : part[i];
        a4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << b0);
    }
    const bool h1 = (lane >> b1) & 1;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = h1 ? a4[i] : a4[i + 2];
        const float keep = h1 ? a4[i + 2] : a4[i];
        a2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << b1);
    }
    const bool h2 = (lane >> b2) & 1;
    float v = (h2 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? a2[0] : a2[1], 1 << b2);
#pragma unroll
    for (int b = b2 - 1; b >= 0; --b) v += __shfl_xor_sync(0xffffffffu, v, 1 << b);
    return v;
}

// Resident CTAs per SM each kernel variant is built for (its register budget).
__host__ __device__ constexpr int decode_ctas_per_sm(int nt, int rt, bool f8 = false) {
    return f8 ? (nt == 1 ? PA_CTAS_PER_SM_F8 : 2)
              : rt == 0 ? (nt == 1 ? PA_CTAS_PER_SM_NT1 : PA_CTAS_PER_SM_NT2) : (rt <= 2 ? 4 : (rt == 4 ? 3 : 2));
}

// Four FP8 E4M3 values (bytes 0..3 of x) widened exactly to two pairs of fp16 values:
// lo = bytes 0, 1 and hi = bytes 2, 3 (the register's 16-bit halves feed the converts directly).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// A pair of bf16 values (one register) as a pair of fp16 values.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
    const float lo = __uint_as_float(x << 16), hi = __uint_as_float(x & 0xffff0000u);
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// NT: query rows per consumer warp / 8 on the tensor-core path (RT == 0).
// RT > 0 selects the CUDA-core path for up to RT (1, 2, 4 or 8) query rows per kv head.
// F8: the K/V caches hold FP8 E4M3 bytes (tensor-core path, fp16 products).
template <typename T, int D, int NT, int RT, bool F8>
__global__ void __launch_bounds__(kThreads, decode_ctas_per_sm(NT, RT, F8))
    decode_kernel(const __grid_constant__ DecodeParams p) {
    using MT = std::conditional_t<F8, __half, T>;  // element type of the tensor-core products
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout lay = smem_layout(D, p.stages, p.mtiles, 8 * NT, p.slot_rows, RT > 0, F8);
    const int qpitch = lay.qpitch;
    constexpr int kRowBytes = D * 2;
    constexpr int kBoxes = D / kBoxCols;  // boxes per K (or V) block
    uint8_t* stage_base = smem;
    uint8_t* qbuf = smem + lay.off_q;
    float* comb_o = reinterpret_cast<float*>(smem + lay.off_comb);
    float* comb_m = reinterpret_cast<float*>(smem + lay.off_m);
    float* comb_l = reinterpret_cast<float*>(smem + lay.off_l);
    UnitInfo* info = reinterpret_cast<UnitInfo*>(smem + lay.off_info);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(info + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_addr(smem + lay.off_bars);
    const uint32_t empty0 = full0 + 8 * kMaxStages;
    const uint32_t qfull0 = empty0 + 8 * kMaxStages;
    const uint32_t qempty0 = qfull0 + 16;
    const int stages = p.stages;
    if (stages < p.block_splits || stages % p.block_splits != 0 || stages > kMaxStages ||
        p.mtiles * p.block_splits != kConsumerWarps) {
        if (threadIdx.x == 0) atomicOr(&g_pa_error, PA_DEVERR_INTERNAL);  // launcher bug: refuse to run
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, p.mtiles);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(qfull0 + 8 * b, 1);
            mbar_init(qempty0 + 8 * b, kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Query rows past `rows` in the last row tile must read as zeros.
    for (int i = threadIdx.x; i < 2 * lay.q_half_bytes / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    __syncthreads();

    griddep_launch_dependents();  // the merge kernel may be scheduled as CTAs retire
    griddep_wait();               // the work list (and the appended K/V) must be complete
    const int units_per_entry = p.num_kv_heads * p.row_groups;  // row groups of one kv head adjacent
    const long long total_units = (long long)p.header[0] * units_per_entry;

    if (warp == kConsumerWarps) {
        // ===================== producer warp =====================
        const uint64_t pol_stream = l2_policy_evict_first();
        const uint64_t pol_keep = l2_policy_evict_last();
        uint32_t k = 0;
        int ul = 0;
        bool ok = true;
        // Units are handed out dynamically, largest first.  The next unit's number, its
        // work entry and its first 32 block ids are fetched while the current unit
        // streams, so a unit starts without dependent loads.
        long long u = 0;
        if (lane == 0) u = atomicAdd(p.work_counter, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        int4 cur = make_int4(0, 0, 0, 0);
        int bids = 0;
        if (u < total_units) {
            cur = p.units[u / units_per_entry];
            const int nb0 = ((min(p.partition, cur.z - cur.y)) + kBlock - 1) / kBlock;
            if (lane < nb0)
                bids = __ldg(p.block_tables + (long long)cur.x * p.max_blocks_per_seq + cur.y / kBlock + lane);
        }
        for (; ok; ++ul) {
            const int qb = ul & 1;
            if (ul >= 2 &&
                !__all_sync(0xffffffffu, mbar_wait(qempty0 + 8 * qb, ((ul - 2) >> 1) & 1, &g_pa_error, abort_flag, p.wait_limit_ns))) {
                ok = false;
                break;
            }
            if (u >= total_units) {  // no work left: hand the consumers an end marker
                if (lane == 0) {
                    info[qb].seq = -1;
                    mbar_arrive(qfull0 + 8 * qb);
                }
                ++ul;
                break;
            }
            const int rem = (int)(u % units_per_entry);
            const int kvh = rem / p.row_groups;
            const int row0 = (rem - kvh * p.row_groups) * p.rows;
            const int nrows = min(p.rows, p.total_rows - row0);
            const int seq = cur.x, tok0 = cur.y, L = cur.z;
            const int ntok = min(p.partition, L - tok0);
            const int nblk = (ntok + kBlock - 1) / kBlock;
            // Next unit: its number is requested now and read two blocks later, its entry is
            // loaded then and its block ids two blocks after that, so no step waits.
            int un_req = 0;
            if (lane == 0) un_req = atomicAdd(p.work_counter, 1);
            long long un = total_units;
            int4 nxt = make_int4(0, 0, 0, 0);
            int nbids = 0;
            if (lane == 0) {
                UnitInfo ui;
                ui.seq = seq;
                ui.tok0 = tok0;
                ui.len = L;
                ui.slot = cur.w;
                ui.kvh = kvh;
                ui.ntok = ntok;
                ui.row0 = row0;
                ui.nrows = nrows;
                info[qb] = ui;
                mbar_arrive_expect_tx(qfull0 + 8 * qb, nrows * kRowBytes);
            }
            __syncwarp();
            for (int r = lane; r < nrows; r += 32) {
                const int qi = (row0 + r) / p.group, hg = (row0 + r) - qi * p.group;
                const T* src = static_cast<const T*>(p.query) +
                               ((long long)(seq * p.q_len + qi) * p.num_heads + kvh * p.group + hg) * D;
                bulk_g2s(smem_addr(qbuf + qb * lay.q_half_bytes + r * qpitch), src, kRowBytes, qfull0 + 8 * qb,
                         pol_keep);
            }
            const int* bt = p.block_tables + (long long)seq * p.max_blocks_per_seq + tok0 / kBlock;
            const int next_at = min(nblk, 2) - 1;      // read the next unit's number, load its entry
            const int prefetch_at = min(nblk, 4) - 1;  // load its first 32 block ids
            for (int c = 0; c < nblk && ok; c += 32) {
                const bool have = c + lane < nblk;
                const int bid = c == 0 ? bids : (have ? __ldg(bt + c + lane) : 0);
                const bool bad = have && (bid < 0 || (long long)bid >= p.num_blocks);
                if (bad) atomicOr(&g_pa_error, PA_DEVERR_BLOCK_ID);
                const int cn = min(32, nblk - c);
                for (int jj = 0; jj < cn; ++jj, ++k) {
                    const int j = c + jj;
                    const int s = (int)(k % stages);
                    if (k >= (uint32_t)stages &&
                        !__all_sync(0xffffffffu,
                                    mbar_wait(empty0 + 8 * s, ((k / stages) - 1) & 1, &g_pa_error, abort_flag, p.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    const int b = __shfl_sync(0xffffffffu, bid, jj);
                    const bool b_bad = __shfl_sync(0xffffffffu, (int)bad, jj) != 0;
                    const int valid = min(kBlock, ntok - kBlock * j);
                    if (lane == 0) {
                        const uint32_t bar = full0 + 8 * s;
                        if (b_bad) {
                            mbar_arrive(bar);  // nothing to wait for; the consumers compute on stale data
                        } else if constexpr (F8) {
                            mbar_arrive_expect_tx(bar, 2 * kBlock * D);
                            const uint32_t dst = smem_addr(stage_base + s * lay.stage_bytes);
                            const int y0 = valid - kBlock;  // <= 0; rows before token 0 arrive as zeros
                            tma_load_4d(dst, &p.tmap_k, 0, kvh, y0, b, bar, pol_stream);
                            tma_load_4d(dst + kBlock * D, &p.tmap_v, 0, kvh, y0, b, bar, pol_stream);
                        } else {
                            mbar_arrive_expect_tx(bar, 2 * kBoxes * kBoxBytes);
                            const uint32_t dst = smem_addr(stage_base + s * lay.stage_bytes);
                            const int y0 = valid - kBlock;  // <= 0; rows before token 0 arrive as zeros
#pragma unroll
                            for (int bx = 0; bx < kBoxes; ++bx) {
                                tma_load_4d(dst + bx * kBoxBytes, &p.tmap_k, bx * kBoxCols, kvh, y0, b, bar,
                                            pol_stream);
                                tma_load_4d(dst + (kBoxes + bx) * kBoxBytes, &p.tmap_v, bx * kBoxCols, kvh, y0, b,
                                            bar, pol_stream);
                            }
                        }
                    }
                    if (c == 0 && jj == next_at) {
                        un = __shfl_sync(0xffffffffu, un_req, 0);
                        if (un < total_units) nxt = p.units[un / units_per_entry];
                    }
                    if (c == 0 && jj == prefetch_at && un < total_units) {
                        const int nb1 = (min(p.partition, nxt.z - nxt.y) + kBlock - 1) / kBlock;
                        if (lane < nb1)
                            nbids = __ldg(p.block_tables + (long long)nxt.x * p.max_blocks_per_seq + nxt.y / kBlock +
                                          lane);
                    }
                }
            }
            // Pad the unit to a multiple of block_splits stages with data-free ones, so every
            // unit starts at a stage counter divisible by block_splits: block j of a unit is
            // then always computed by warp j % block_splits, whichever CTA gets the unit, and
            // the result does not depend on the order in which units are handed out.
            const int nblk_pad = ((nblk + p.block_splits - 1) / p.block_splits) * p.block_splits;
            for (int j = nblk; j < nblk_pad && ok; ++j, ++k) {
                const int s = (int)(k % stages);
                if (k >= (uint32_t)stages &&
                    !__all_sync(0xffffffffu,
                                mbar_wait(empty0 + 8 * s, ((k / stages) - 1) & 1, &g_pa_error, abort_flag, p.wait_limit_ns))) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive(full0 + 8 * s);
                __syncwarp();
            }
            cur = nxt;
            bids = nbids;
            u = un;
        }
        // Never leave the CTA with copies in flight: wait for the last fill of every
        // stage and of both query buffers (immediate on the normal path).
        for (int s = 0; s < stages; ++s) {
            if (k > (uint32_t)s) {
                const uint32_t last = s + ((k - 1 - s) / stages) * stages;
                mbar_wait(full0 + 8 * s, (last / stages) & 1, &g_pa_error, nullptr);
            }
        }
        for (int back = 1; back <= 2; ++back) {
            const int u2 = ul - back;
            if (u2 >= 0) mbar_wait(qfull0 + 8 * (u2 & 1), (u2 >> 1) & 1, &g_pa_error, nullptr);
        }
        return;
    }

    // ===================== consumer warps =====================
    // Transposed tiles, so that the few query rows of a kv head fill the N side of
    // the m16n8k16 tensor-core tile instead of padding its M side:
    //   S^T  = K Q^T     M = 16 tokens,      N = 8 query rows, K = head dim
    //   O^T += V^T P^T   M = 16 head-dim cols, N = 8 query rows, K = 16 tokens
    // Each warp owns NT groups of 8 query rows (one row tile) and every
    // block_splits-th block of the unit.
    constexpr int TR = 8 * NT;               // query rows per warp (8 on the CUDA-core path)
    const int mt = warp / p.block_splits;   // row tile of this warp
    const int bsg = warp % p.block_splits;  // which of the tile's block-split warps
    const int gid = lane >> 2, tig = lane & 3;
    uint32_t k = 0;
    int ul = 0;
    for (;; ++ul) {
        const int qb = ul & 1;
        // (all waits below are made warp-uniform: a timeout seen by one lane stops the warp)
        bool ok = __all_sync(0xffffffffu, mbar_wait(qfull0 + 8 * qb, (ul >> 1) & 1, &g_pa_error, abort_flag, p.wait_limit_ns));
        const UnitInfo ui = info[qb];
        const bool done = ok && ui.seq < 0;  // end marker: no unit follows
        const int rows_here = min(TR, ui.nrows - mt * TR);  // <= 0 for an all-padding tile
        if constexpr (RT == 0) {
            uint32_t qf[NT][D / 16][2];      // Q^T as the B operand: Q[row][d 2t..2t+1], Q[row][d 2t+8..2t+9]
            float m[NT][2], l[NT][2];        // running max (log2 units) and sum for rows 2t, 2t+1 of each group
            float o[D / 16][NT][4];          // O^T: (d gid, row 2t), (d gid, row 2t+1), (d gid+8, 2t), (d gid+8, 2t+1)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                m[nt][0] = m[nt][1] = -INFINITY;
                l[nt][0] = l[nt][1] = 0.f;
            }
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) o[dt][nt][0] = o[dt][nt][1] = o[dt][nt][2] = o[dt][nt][3] = 0.f;
            int nblk = 0, nblk_pad = 0;
            if (ok && !done) {
                const uint8_t* qrow = qbuf + qb * lay.q_half_bytes + mt * TR * qpitch;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int k2 = 0; k2 < D / 32; ++k2) {
                        const int rr = nt * 8 + (lane & 7);
                        const int cc = k2 * 32 + (lane >> 3) * 8;
                        ldsm_x4(smem_addr(qrow + rr * qpitch + cc * 2), qf[nt][2 * k2][0], qf[nt][2 * k2][1],
                                qf[nt][2 * k2 + 1][0], qf[nt][2 * k2 + 1][1]);
                    }
                if constexpr (F8) {
                    // Same permuted contraction order as the K fragments: step kk of lane tig
                    // takes query elements tig*32 + kk*4 .. +3; products run in fp16.  A bf16
                    // query is rounded to fp16 (exact for its 8 significant bits down to 2^-17);
                    // an element of magnitude >= 65520 would become infinite, and is refused:
                    // PA_DEVERR_QUERY_RANGE, that row's output undefined (each query row is its
                    // own column of the products, so the other rows are unaffected).
                    float amax = 0.f;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint8_t* qr = qrow + (nt * 8 + gid) * qpitch + tig * 64;
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const uint4 x = *reinterpret_cast<const uint4*>(qr + c4 * 16);
                            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t r0 = w4[2 * h], r1 = w4[2 * h + 1];
                                if constexpr (Elem<T>::kDtype == PA_BF16) {
                                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(r0 << 16)), fabsf(__uint_as_float(r0 & 0xffff0000u))),
                                                             fmaxf(fabsf(__uint_as_float(r1 << 16)), fabsf(__uint_as_float(r1 & 0xffff0000u)))));
                                    r0 = bf16x2_to_f16x2(r0);
                                    r1 = bf16x2_to_f16x2(r1);
                                }
                                qf[nt][c4 * 2 + h][0] = r0;
                                qf[nt][c4 * 2 + h][1] = r1;
                            }
                        }
                    }
                    if (Elem<T>::kDtype == PA_BF16 && __any_sync(0xffffffffu, amax >= 65520.f) && lane == 0)
                        atomicOr(&g_pa_error, PA_DEVERR_QUERY_RANGE);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8 * qb);

                nblk = (ui.ntok + kBlock - 1) / kBlock;
                nblk_pad = ((nblk + p.block_splits - 1) / p.block_splits) * p.block_splits;
                const int tok0 = ui.tok0;
                // Last position (relative to the partition) each of this lane's rows may see:
                // row j of the q_len-row chunk is position L - q_len + j.
                int lim[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int r = ui.row0 + mt * TR + nt * 8 + 2 * tig + c;
                        lim[nt][c] = ui.len - p.q_len + min(r / p.group, p.q_len - 1) - tok0;
                    }
                int lim_lo = lim[0][0];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) lim_lo = min(lim_lo, min(lim[nt][0], lim[nt][1]));
                // Units start at a stage counter divisible by block_splits (the producer pads
                // them), so this warp's blocks are j = bsg, bsg + block_splits, ...
                for (int j = bsg; j < nblk_pad; j += p.block_splits) {
                    const uint32_t kj = k + j;
                    const int s = (int)(kj % stages);
                    if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (kj / stages) & 1, &g_pa_error, abort_flag, p.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    // Data-free padding stages are only waited for and released, and so is every stage
                    // by a warp whose row tile holds only padding rows (a third row tile rounded up to
                    // four): its results are never read.
                    if (j < nblk && rows_here > 0) {
                        const uint32_t kst = smem_addr(stage_base + s * lay.stage_bytes);
                        const uint32_t vst = kst + kBoxes * kBoxBytes;
                        // smem row i holds token i - shift of this block (shift > 0 only for a short last block)
                        const int shift = kBlock - min(kBlock, ui.ntok - kBlock * j);
                        float sc[NT][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                        if constexpr (F8) {
                            // FP8 stage, 128 B rows, 128-byte swizzled.  The head-dim order of the
                            // contraction is permuted (Q's fragments follow it): the lane's four
                            // k columns of step kk are bytes t*32 + kk*4 .. +3 of its token rows, so
                            // each register is one adjacent E4M3 pair widened to fp16.
                            const uint8_t* k8 = stage_base + s * lay.stage_bytes;
                            // Even and odd k-steps into two accumulators, summed at the end: half the
                            // chain of dependent products (same-box A/B 131.6-131.9 vs 132.5 us).
                            float sc2[NT][4];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) sc2[nt][0] = sc2[nt][1] = sc2[nt][2] = sc2[nt][3] = 0.f;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint4 lo = *reinterpret_cast<const uint4*>(
                                    k8 + gid * 128 + ((((tig * 2 + h) ^ (gid & 7))) << 4));
                                const uint4 hi = *reinterpret_cast<const uint4*>(
                                    k8 + (gid + 8) * 128 + ((((tig * 2 + h) ^ ((gid + 8) & 7))) << 4));
                                const uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
                                const uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                                for (int q4 = 0; q4 < 4; ++q4) {
                                    const int kk = h * 4 + q4;
                                    uint32_t a[4];
                                    e4m3x4_to_f16x2x2(wl[q4], a[0], a[2]);
                                    e4m3x4_to_f16x2x2(wh[q4], a[1], a[3]);
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt)
                                        Elem<MT>::mma((kk & 1) ? sc2[nt] : sc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                                }
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 4; ++c) sc[nt][c] += sc2[nt][c];
                        } else {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                uint32_t a[4];
                                const int tr = (lane & 7) + ((lane >> 3) & 1) * 8;
                                const int cc = kk * 16 + (lane >> 4) * 8;
                                ldsm_x4(kst + swz(tr, cc), a[0], a[1], a[2], a[3]);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) Elem<MT>::mma(sc[nt], a, qf[nt][kk][0], qf[nt][kk][1]);
                            }
                        }
                        constexpr bool kLazy = ((PA_LAZY_MAX >> (F8 ? 0 : 1)) & 1) != 0;
                        // Scale into log2 units; mask positions past each row's limit (and the zero rows
                        // in front of a short block).  A block whose every position all of the lane's rows
                        // may see needs no mask.
                        if (kLazy && shift == 0 && kBlock * j + kBlock - 1 <= lim_lo) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 4; ++c) sc[nt][c] *= p.scale_log2;
                        } else {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const int i = gid + (c >> 1) * 8;
                                    const int tok = kBlock * j + i - shift;
                                    sc[nt][c] = (i >= shift && tok <= lim[nt][c & 1]) ? sc[nt][c] * p.scale_log2 : -INFINITY;
                                }
                        }
                        float pr[NT][4];
                        if constexpr (kLazy) {
                            // The running max m moves only when some score of the warp's rows passes it by
                            // more than 8 (weights up to 2^8 otherwise), found by one vote: most blocks
                            // skip the cross-lane max and the rescale of O.  m stays the same in the eight
                            // lanes holding a row, so the weights, l and O keep one reference per row.
                            bool bump = false;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 2; ++c) bump |= fmaxf(sc[nt][c], sc[nt][c + 2]) > m[nt][c] + 8.f;
                            if (__any_sync(0xffffffffu, bump)) {
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                    for (int c = 0; c < 2; ++c) {
                                        float mx = fmaxf(sc[nt][c], sc[nt][c + 2]);
                                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                                        const float mn = fmaxf(m[nt][c], mx);
                                        const float a = ex2(m[nt][c] - (mn == -INFINITY ? 0.f : mn));
                                        m[nt][c] = mn;
                                        l[nt][c] *= a;
#pragma unroll
                                        for (int dt = 0; dt < D / 16; ++dt) {
                                            o[dt][nt][c] *= a;
                                            o[dt][nt][c + 2] *= a;
                                        }
                                    }
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                for (int c = 0; c < 2; ++c) {
                                    const float base = m[nt][c] == -INFINITY ? 0.f : m[nt][c];
                                    pr[nt][c] = ex2(sc[nt][c] - base);
                                    pr[nt][c + 2] = ex2(sc[nt][c + 2] - base);
                                    l[nt][c] += pr[nt][c] + pr[nt][c + 2];
                                }
                        } else {
                        float alpha[NT][2];
                        bool rescale = false;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                float mx = fmaxf(sc[nt][c], sc[nt][c + 2]);
                                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                                const float mn = fmaxf(m[nt][c], mx);
                                const float base = mn == -INFINITY ? 0.f : mn;
                                alpha[nt][c] = ex2(m[nt][c] - base);
                                rescale |= alpha[nt][c] != 1.f;
                                m[nt][c] = mn;
                                pr[nt][c] = ex2(sc[nt][c] - base);
                                pr[nt][c + 2] = ex2(sc[nt][c + 2] - base);
                                l[nt][c] = l[nt][c] * alpha[nt][c] + (pr[nt][c] + pr[nt][c + 2]);
                            }
                        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                            for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    o[dt][nt][0] *= alpha[nt][0];
                                    o[dt][nt][1] *= alpha[nt][1];
                                    o[dt][nt][2] *= alpha[nt][0];
                                    o[dt][nt][3] *= alpha[nt][1];
                                }
                        }
                        }
                        // P^T as the B operand, in two 16-bit pieces (hi + residual) that together carry
                        // about 16 significant bits.  The lane's (token, row-pair) values form the standard
                        // fragment of P^T's 8x8 sub-tiles; movmatrix transposes them into (row, token-pair).
                        uint32_t pb_hi[NT][2], pb_lo[NT][2];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const float x0 = pr[nt][2 * h], x1 = pr[nt][2 * h + 1];
                                if constexpr (F8) {
                                    pb_hi[nt][h] = movmatrix_trans(Elem<MT>::pack(x0, x1));
                                } else {
                                    const float h0 = Elem<MT>::round_trip(x0), h1 = Elem<MT>::round_trip(x1);
                                    pb_hi[nt][h] = movmatrix_trans(Elem<MT>::pack(h0, h1));
                                    pb_lo[nt][h] = movmatrix_trans(Elem<MT>::pack(x0 - h0, x1 - h1));
                                }
                            }
                        if constexpr (F8) {
                            // Output columns are permuted inside each 16-column tile: tile dt's rows
                            // gid and gid+8 are head-dim columns gid*16 + 2dt and +1, so the lane
                            // needs bytes gid*16 .. +15 of its four token rows 2t, 2t+1, 2t+8, 2t+9;
                            // a byte permute pairs the two tokens of each column.
                            const uint8_t* v8 = stage_base + s * lay.stage_bytes + kBlock * D;
                            uint32_t vw[4][4];
#pragma unroll
                            for (int rr = 0; rr < 4; ++rr) {
                                const int r = 2 * tig + (rr & 1) + (rr >> 1) * 8;
                                const uint4 x = *reinterpret_cast<const uint4*>(v8 + r * 128 + ((gid ^ (r & 7)) << 4));
                                vw[rr][0] = x.x;
                                vw[rr][1] = x.y;
                                vw[rr][2] = x.z;
                                vw[rr][3] = x.w;
                            }
                            __syncwarp();
                            if (lane == 0) mbar_arrive(empty0 + 8 * s);  // stage consumed: everything is in registers
#pragma unroll
                            for (int dt = 0; dt < D / 16; ++dt) {
                                const int w = dt >> 1, b = (dt & 1) * 2;
                                const uint32_t sel = b | (4 + b) << 4 | (b + 1) << 8 | (5 + b) << 12;
                                const uint32_t p01 = __byte_perm(vw[0][w], vw[1][w], sel);  // tokens 2t, 2t+1
                                const uint32_t p89 = __byte_perm(vw[2][w], vw[3][w], sel);  // tokens 2t+8, 2t+9
                                uint32_t a[4];
                                e4m3x4_to_f16x2x2(p01, a[0], a[1]);
                                e4m3x4_to_f16x2x2(p89, a[2], a[3]);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)  // E4M3 V has 4 significant bits: fp16 P suffices
                                    Elem<MT>::mma(o[dt][nt], a, pb_hi[nt][0], pb_hi[nt][1]);
                            }
                        } else {
#pragma unroll
                            for (int dt = 0; dt < D / 16; ++dt) {
                                uint32_t a[4];
                                const int tr = (lane & 7) + (lane >> 4) * 8;
                                const int cc = dt * 16 + ((lane >> 3) & 1) * 8;
                                ldsm_x4_trans(vst + swz(tr, cc), a[0], a[1], a[2], a[3]);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    Elem<MT>::mma(o[dt][nt], a, pb_hi[nt][0], pb_hi[nt][1]);
                                    Elem<MT>::mma(o[dt][nt], a, pb_lo[nt][0], pb_lo[nt][1]);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    // (FP8: a computing warp released the stage right after its loads)
                    if (lane == 0 && !(F8 && j < nblk && rows_here > 0)) mbar_arrive(empty0 + 8 * s);
                }
            }
            k += nblk_pad;
            // Row sums over the eight lanes (same tig) that hold a row's tokens.
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 4);
                    l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 8);
                    l[nt][c] += __shfl_xor_sync(0xffffffffu, l[nt][c], 16);
                }
            if (ok && !done) {
                float* co = comb_o + warp * p.slot_rows * D;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int row = nt * 8 + 2 * tig + c;
                        if (row < rows_here) {
#pragma unroll
                            for (int dt = 0; dt < D / 16; ++dt) {
                                if constexpr (F8) {  // permuted columns: gid*16 + 2dt and + 1
                                    *reinterpret_cast<float2*>(co + row * D + gid * 16 + dt * 2) =
                                        make_float2(o[dt][nt][c], o[dt][nt][c + 2]);
                                } else {
                                    co[row * D + dt * 16 + gid] = o[dt][nt][c];
                                    co[row * D + dt * 16 + gid + 8] = o[dt][nt][c + 2];
                                }
                            }
                            if (gid == 0) {
                                comb_m[warp * kCombRows + row] = m[nt][c];
                                comb_l[warp * kCombRows + row] = l[nt][c];
                            }
                        }
                    }
            }
        } else {
            // ---------- CUDA-core path: fp32 FMA dot products and warp-shuffle reductions ----------
            // Lane = (column chunk c of 8 head-dim elements, token parity tp).  For every token
            // the lane forms partial dot products of its 8 columns with all RT query rows; a
            // transposing butterfly over the CH lanes of the row leaves each lane holding the
            // full score of one row rr.  P and the rescale factors are exchanged through shared
            // memory for P.V, which every lane accumulates for all rows over its 8 columns.
            constexpr int CH = D / 8, TPI = 32 / CH, ITERS = kBlock / TPI;
            constexpr int LCH = D == 128 ? 4 : 3;
            const int c = lane % CH, tp = lane / CH;
            const int rr = (c >> (LCH - 3)) & 7;
            const bool row_owner = LCH == 3 || (c & 1) == 0;
            float* pbuf = reinterpret_cast<float*>(smem + lay.off_fma) + warp * kFmaWarpFloats;
            float qv[RT][8], o[RT][8];
            float m_r = -INFINITY, l_r = 0.f;
#pragma unroll
            for (int r = 0; r < RT; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[r][e] = 0.f;
            int nblk = 0, nblk_pad = 0;
            if (ok && !done) {
                const uint8_t* qrow = qbuf + qb * lay.q_half_bytes;
#pragma unroll
                for (int r = 0; r < RT; ++r) unpack8<T>(*reinterpret_cast<const uint4*>(qrow + r * qpitch + c * 16), qv[r]);
                __syncwarp();
                if (lane == 0) mbar_arrive(qempty0 + 8 * qb);
                nblk = (ui.ntok + kBlock - 1) / kBlock;
                nblk_pad = ((nblk + p.block_splits - 1) / p.block_splits) * p.block_splits;
                const int lim_r = ui.len - p.q_len + min((ui.row0 + rr) / p.group, p.q_len - 1) - ui.tok0;
                for (int j = bsg; j < nblk_pad; j += p.block_splits) {
                    const uint32_t kj = k + j;
                    const int s = (int)(kj % stages);
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(full0 + 8 * s, (kj / stages) & 1, &g_pa_error, abort_flag, p.wait_limit_ns))) {
                        ok = false;
                        break;
                    }
                    if (j < nblk) {
                        const uint8_t* kst = stage_base + s * lay.stage_bytes;
                        const uint8_t* vst = kst + (D / kBoxCols) * kBoxBytes;
                        const int shift = kBlock - min(kBlock, ui.ntok - kBlock * j);
                        float sv[ITERS];
#pragma unroll
                        for (int it = 0; it < ITERS; ++it) {
                            const int i = it * TPI + tp;
                            float kf[8], part[8];
                            unpack8<T>(*reinterpret_cast<const uint4*>(kst + swz(i, c * 8)), kf);
#pragma unroll
                            for (int r = 0; r < 8; ++r) {
                                float acc = 0.f;
                                if (r < RT) {
#pragma unroll
                                    for (int e = 0; e < 8; ++e) acc = fmaf(qv[r < RT ? r : 0][e], kf[e], acc);
                                }
                                part[r] = acc;
                            }
                            sv[it] = transpose_reduce8<LCH>(part, lane);
                        }
                        float mx = -INFINITY;
#pragma unroll
                        for (int it = 0; it < ITERS; ++it) {
                            const int i = it * TPI + tp;
                            const int tok = kBlock * j + i - shift;
                            sv[it] = (i >= shift && tok <= lim_r) ? sv[it] * p.scale_log2 : -INFINITY;
                            mx = fmaxf(mx, sv[it]);
                        }
#pragma unroll
                        for (int o2 = CH; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
                        const float mn = fmaxf(m_r, mx);
                        const float base = mn == -INFINITY ? 0.f : mn;
                        const float alpha = ex2(m_r - base);
                        m_r = mn;
                        float psum = 0.f;
#pragma unroll
                        for (int it = 0; it < ITERS; ++it) {
                            sv[it] = ex2(sv[it] - base);
                            psum += sv[it];
                        }
                        l_r = l_r * alpha + psum;
                        if (row_owner) {
#pragma unroll
                            for (int it = 0; it < ITERS; ++it) pbuf[rr * 16 + tp * ITERS + it] = sv[it];
                            if (tp == 0) pbuf[128 + rr] = alpha;
                        }
                        __syncwarp();
                        bool rescale = false;
                        float al[RT];
#pragma unroll
                        for (int r = 0; r < RT; ++r) {
                            al[r] = pbuf[128 + r];
                            rescale |= al[r] != 1.f;
                        }
                        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                            for (int r = 0; r < RT; ++r)
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[r][e] *= al[r];
                        }
#pragma unroll
                        for (int it = 0; it < ITERS; ++it) {
                            const int i = it * TPI + tp;
                            float vf[8];
                            unpack8<T>(*reinterpret_cast<const uint4*>(vst + swz(i, c * 8)), vf);
#pragma unroll
                            for (int r = 0; r < RT; ++r) {
                                const float pr = pbuf[r * 16 + tp * ITERS + it];
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[r][e] = fmaf(pr, vf[e], o[r][e]);
                            }
                        }
                        __syncwarp();  // pbuf is rewritten by the next block
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty0 + 8 * s);
                }
            }
            k += nblk_pad;
            // Sum over the token-parity lanes.
#pragma unroll
            for (int o2 = CH; o2 < 32; o2 <<= 1) {
                l_r += __shfl_xor_sync(0xffffffffu, l_r, o2);
#pragma unroll
                for (int r = 0; r < RT; ++r)
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[r][e] += __shfl_xor_sync(0xffffffffu, o[r][e], o2);
            }
            if (ok && !done) {
                float* co = comb_o + warp * p.slot_rows * D;
                if (tp == 0) {
#pragma unroll
                    for (int r = 0; r < RT; ++r)
                        if (r < rows_here) {
                            *reinterpret_cast<float4*>(co + r * D + c * 8) = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
                            *reinterpret_cast<float4*>(co + r * D + c * 8 + 4) = make_float4(o[r][4], o[r][5], o[r][6], o[r][7]);
                        }
                    if (row_owner && rr < rows_here) {
                        comb_m[warp * kCombRows + rr] = m_r;
                        comb_l[warp * kCombRows + rr] = l_r;
                    }
                }
            }
        }
        // All consumer warps agree on whether to go on (and the buffer writes above are
        // ordered before the reads below).
        if (consumers_any(!ok || done)) break;
        // Merge the block-split warps of each row tile; write the output or the partial.
        const int nthreads = kConsumerWarps * 32;
        for (int idx = threadIdx.x; idx < ui.nrows * D; idx += nthreads) {
            const int r = idx / D, e = idx - r * D;
            const int tile = r / TR, rr = r - tile * TR;
            float M = -INFINITY;
            for (int b = 0; b < p.block_splits; ++b) M = fmaxf(M, comb_m[(tile * p.block_splits + b) * kCombRows + rr]);
            float lsum = 0.f, acc = 0.f;
            if (M != -INFINITY) {
                for (int b = 0; b < p.block_splits; ++b) {
                    const int w = tile * p.block_splits + b;
                    const float f = ex2(comb_m[w * kCombRows + rr] - M);
                    lsum += comb_l[w * kCombRows + rr] * f;
                    acc += comb_o[(w * p.slot_rows + rr) * D + e] * f;
                }
            }
            const int qi = (ui.row0 + r) / p.group;
            const int h = ui.kvh * p.group + (ui.row0 + r - qi * p.group);
            const long long orow = (long long)(ui.seq * p.q_len + qi) * p.num_heads + h;
            if (ui.slot < 0) {
                static_cast<uint16_t*>(p.out)[orow * D + e] = Elem<T>::to_bits(acc * p.v_scale / lsum);
            } else {
                const long long prow = ((long long)ui.slot * p.q_len + qi) * p.num_heads + h;
                p.pacc[prow * D + e] = acc * p.v_scale;
                if (e == 0) p.pml[prow] = make_float2(M, lsum);
            }
        }
        named_barrier_sync(1, nthreads);
    }
}

// ---------------------------------------------------------------------------
// Split-K merge
// ---------------------------------------------------------------------------
struct MergeParams {
    void* out;
    const int* part_start;
    const float2* pml;
    const float* pacc;
    int num_seqs;
    int q_len;
    int num_heads;
};

// One warp per output row (sequence, query row, head) of a sequence with more than one
// piece (part_start[i + 1] - part_start[i] partial results: split-K partitions, and a shared
// prefix's piece first).  The pieces' (max, sum) pairs are read lane-parallel and turned into
// weights e^{m_p - M} / sum_p' e^{m_p' - M} l_p' once; the unnormalised partial outputs are
// then summed in slot order, so the result does not depend on timing.  Sequences with one
// piece (written by the partition pass) or none (an invalid length) are skipped.
template <typename T, int D>
__device__ __forceinline__ void merge_body(const MergeParams& p, const PrefixGroups* g) {
    constexpr int kPer = D / 32;
    const long long row = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows_total = (long long)p.num_seqs * p.q_len * p.num_heads;
    if (row >= rows_total) return;
    const int per_seq = p.q_len * p.num_heads;
    const int seq = (int)(row / per_seq);
    const int rem = (int)(row - (long long)seq * per_seq);
    const long long slot0 = p.part_start[seq];
    const int nparts = p.part_start[seq + 1] - (int)slot0;
    if (nparts <= 1) return;
    if (g && prefix_of(*g, seq) > 0) return;  // finished by the shared-prefix kernel
    // Lane l keeps the (max, sum) pairs of partitions l and l + 32; any further ones are re-read.
    const float2 ml0 = lane < nparts ? p.pml[(slot0 + lane) * per_seq + rem] : make_float2(-INFINITY, 0.f);
    const float2 ml1 = lane + 32 < nparts ? p.pml[(slot0 + lane + 32) * per_seq + rem] : make_float2(-INFINITY, 0.f);
    float M = fmaxf(ml0.x, ml1.x);
    for (int i = lane + 64; i < nparts; i += 32) M = fmaxf(M, p.pml[(slot0 + i) * per_seq + rem].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float lsum = 0.f;
    if (lane < nparts) lsum += ml0.y * ex2(ml0.x - M);
    if (lane + 32 < nparts) lsum += ml1.y * ex2(ml1.x - M);
    for (int i = lane + 64; i < nparts; i += 32) {
        const float2 ml = p.pml[(slot0 + i) * per_seq + rem];
        lsum += ml.y * ex2(ml.x - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    float acc[kPer];
#pragma unroll
    for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
    for (int base = 0; base < nparts; base += 32) {
        const int mine = base + lane;
        const float m_mine = base == 0 ? ml0.x : base == 32 ? ml1.x
                                                             : (mine < nparts ? p.pml[(slot0 + mine) * per_seq + rem].x : 0.f);
        const float f_mine = mine < nparts ? ex2(m_mine - M) * inv : 0.f;
        const int cnt = min(32, nparts - base);
#pragma unroll 8
        for (int j = 0; j < cnt; ++j) {
            const float f = __shfl_sync(0xffffffffu, f_mine, j);
            const float* src = p.pacc + ((slot0 + base + j) * per_seq + rem) * D + lane * kPer;
            if constexpr (kPer == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] += v.x * f;
                acc[1] += v.y * f;
                acc[2] += v.z * f;
                acc[3] += v.w * f;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] += v.x * f;
                acc[1] += v.y * f;
            }
        }
    }
    uint16_t* dst = static_cast<uint16_t*>(p.out) + row * D + lane * kPer;
#pragma unroll
    for (int c = 0; c < kPer; ++c) dst[c] = Elem<T>::to_bits(acc[c]);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
    griddep_launch_dependents();  // the next call's append may be scheduled; it waits for this grid
    griddep_wait();               // the partition pass must have finished
    merge_body<T, D>(p, nullptr);
}

// After a shared-prefix call's prefix kernel (which merges its own sequences): the others.
template <typename T, int D>
__global__ void __launch_bounds__(128) merge_ungrouped_kernel(const MergeParams p, const __grid_constant__ PrefixGroups g) {
    griddep_launch_dependents();
    griddep_wait();
    merge_body<T, D>(p, &g);
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
namespace {

std::mutex g_mu;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int max_smem_optin = 0;
};
DeviceInfo g_dev[64];

int device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        d.ready = true;
    }
    out = d;
    return PA_OK;
}

// Occupancy of one decode instantiation for a given dynamic shared memory size,
// cached per device.
struct OccEntry {
    const void* fn;
    int dev, smem, blocks;
};
OccEntry g_occ[256];
int g_occ_n = 0;

int decode_blocks_per_sm(const void* fn, int smem, int& blocks) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_occ_n; ++i)
        if (g_occ[i].fn == fn && g_occ[i].dev == dev && g_occ[i].smem == smem) {
            blocks = g_occ[i].blocks;
            return PA_OK;
        }
    // The opt-in limit is raised to what this call needs and never lowered, so every
    // cached (fn, smem) entry stays launchable.
    int cur = 0;
    {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return PA_ERR_CUDA;
        cur = fa.maxDynamicSharedSizeBytes;
    }
    if (cur < smem && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PA_ERR_CUDA;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, kThreads, smem) != cudaSuccess) return PA_ERR_CUDA;
    if (b < 1) return PA_ERR_UNSUPPORTED;
    if (g_occ_n < 256) g_occ[g_occ_n++] = OccEntry{fn, dev, smem, b};
    blocks = b;
    return PA_OK;
}

// 0: auto, 1: CUDA-core FMA (up to 8 rows per kv head), 2: mma.sync tensor-core tiles,
// 3: the tcgen05 prefill kernel for every call over 16-bit caches
int g_decode_math = 0;

// Benchmark timing marks of each decode call: 0 before the plan kernel, 1 before the main
// kernel (the split-K partition pass or the tcgen05 kernel), 2 after it, 3 after the merge.
// In mode 2 mark 2 is not recorded, so nothing separates the main kernel from the merge kernel
// (their programmatic overlap is kept) and the main figure covers both.
constexpr int kProfCalls = 2048;
struct Profile {
    int mode = 0;  // 0 off, 1 every mark, 2 marks 0, 1 and 3
    int dev = -1;
    int n = 0;
    cudaEvent_t ev[4 * kProfCalls] = {};
    bool created = false;
} g_prof;

// cuTensorMapEncodeTiled, fetched from the driver at first use (no link-time libcuda dependency).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// The pool [num_blocks, 16, Hkv, D] as a 4-D tensor (innermost first: D, Hkv, 16, num_blocks);
// one box = 64 elements of one kv head for the 16 tokens of one block, 128-byte swizzled.
int make_kv_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks, int num_kv_heads, int head_dim) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)kBlock,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_kv_heads * head_dim * 2,
                                   (cuuint64_t)kBlock * num_kv_heads * head_dim * 2};
    const cuuint32_t box[4] = {(cuuint32_t)kBoxCols, 1, (cuuint32_t)kBlock, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_INVALID_ARG;
}

// An FP8 pool [num_blocks, 16, Hkv, D] bytes: one box = the 16 rows (128 B) of one kv head, 128-byte swizzled.
int make_kv_map_fp8(CUtensorMap* map, const void* base, int64_t num_blocks, int num_kv_heads, int head_dim) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return PA_ERR_CUDA;
    const cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads, (cuuint64_t)kBlock,
                                (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_kv_heads * head_dim,
                                   (cuuint64_t)kBlock * num_kv_heads * head_dim};
    const cuuint32_t box[4] = {(cuuint32_t)head_dim, 1, (cuuint32_t)kBlock, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_INVALID_ARG;
}

// Consumer arithmetic of the decode kernel for `rows` query rows per work unit: rt > 0 picks the
// CUDA-core path for up to rt rows, else tensor-core tiles with warps of 8 * nt rows.
// Measured on GB300 (partition kernel, CUDA events): with one query row per kv head both paths
// stream at the same rate (MHA workload 6.33 vs 6.35 TB/s), so that case stays on CUDA-core FMA;
// with grouped heads the tensor-core tiles win (4 rows: 5.99 vs 3.79 TB/s, 8 rows: 5.88 vs
// 1.91 TB/s).
void decode_variant(int rows, bool fp8, int& rt, int& nt) {
    rt = 0;
    if (g_decode_math == 1 && rows <= 8) rt = rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
    if (g_decode_math == 0 && rows == 1) rt = 1;
    if (fp8) rt = 0;  // FP8 caches are read on the tensor-core path
    nt = (rows <= 8 || (PA_PREFER_NT1 && rows <= 32)) ? 1 : 2;
}

// Split-K partition when the caller leaves it to the library: the largest of 512, 1024 and 2048
// tokens that still gives about three work units per resident CTA, counting each sequence as
// max_context_len / 2 positions long.  Larger partitions leave fewer fp32 partials to merge;
// the largest-first hand-out keeps the tail short while units are plentiful.  Measured on GB300
// (call time): GQA batch of 128, 512 / 1024 / 2048 tokens: 181.7 / 177.6 / - us; long context
// (16 sequences of 16-32K + 240 short): 408.6 / 376.5 / 357.3 us (4096: 397.9); OPT-13B-shaped
// MHA: 156.2 / 158.7 / 182.4 us; 32 GQA sequences: 68.1 / 68.3 / 92.2 us.  The same rule for an
// FP8 cache; GQA batch of 128, partition kernel, 512 / 1024 / 2048 tokens: 130.5 / 126.5 / 141.3 us.
int auto_partition(const DecodeArgs& a, int sms) {
    const int group = a.num_heads / a.num_kv_heads;
    const long long total_rows = (long long)group * a.q_len;
    const int rows = (int)std::min<long long>(PA_ROW_GROUP_ROWS, total_rows);
    const long long row_groups = (total_rows + rows - 1) / rows;
    int rt, nt;
    decode_variant(rows, a.fp8, rt, nt);
    const long long slots = (long long)sms * decode_ctas_per_sm(nt, rt, a.fp8);
    const long long half = std::max(1, a.max_context_len / 2);
    int best = PA_DEFAULT_PARTITION;
    for (int part = 2 * PA_DEFAULT_PARTITION; part <= 4 * PA_DEFAULT_PARTITION; part *= 2) {
        const long long units = (long long)a.num_seqs * a.num_kv_heads * row_groups * ((half + part - 1) / part);
        if (units >= 3 * slots) best = part;
    }
    return best;
}

// The same choice for a shared-prefix call, over the positions after each group's prefix
// (taken as half of what is left of max_context_len).  Measured on the shared-prefix batch
// (64 sequences, 1024-token prefix, suffixes of 16-512 positions, 20 rows per kv head), step
// time: 64 / 128 / 256 / 512 tokens 98.4 / 83.4 / 76.3 / 73.6 us: every partition costs its CTA
// a fixed set-up and combine, so finer splits of short suffixes lose.
int auto_partition_prefix(const DecodeArgs& a, int sms) {
    const PrefixGroups& g = *a.groups;
    const int group = a.num_heads / a.num_kv_heads;
    const long long total_rows = (long long)group * a.q_len;
    const int rows = (int)std::min<long long>(PA_ROW_GROUP_ROWS, total_rows);
    const long long row_groups = (total_rows + rows - 1) / rows;
    int rt, nt;
    decode_variant(rows, false, rt, nt);
    const long long slots = (long long)sms * decode_ctas_per_sm(nt, rt, false);
    int best = kMinPrefixPartition;
    for (int part = kMinPrefixPartition; part <= 4 * PA_DEFAULT_PARTITION; part *= 2) {
        long long units = 0;
        int grouped = 0;
        for (int k = 0; k < g.n; ++k) {
            const int n_k = g.seq_start[k + 1] - g.seq_start[k];
            const long long rest = std::max(16, (a.max_context_len - g.len[k]) / 2);
            units += (long long)n_k * ((rest + part - 1) / part);
            grouped += n_k;
        }
        const long long half = std::max(1, a.max_context_len / 2);
        units += (long long)(a.num_seqs - grouped) * ((half + part - 1) / part);
        if (units * a.num_kv_heads * row_groups >= 3 * slots) best = part;
    }
    return best;
}

template <typename T, int D>
int launch_decode_typed(const DecodeArgs& a, cudaStream_t stream, int* launches) {
    const bool prefix = a.groups != nullptr;
    const WsLayout w = ws_layout(a.num_seqs, a.q_len, a.num_heads, D, a.max_context_len, a.partition, prefix);
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    int* header = reinterpret_cast<int*>(ws + w.header);
    int* part_start = reinterpret_cast<int*>(ws + w.part_start);
    int4* units = reinterpret_cast<int4*>(ws + w.units);
    float2* pml = reinterpret_cast<float2*>(ws + w.pml);
    float* pacc = reinterpret_cast<float*>(ws + w.pacc);

    DeviceInfo dev;
    if (int st = device_info(dev)) return st;

    const int pc = profile_call_begin();
    profile_mark(pc, 0, stream);
    PlanParams pp;
    pp.context_lens = a.context_lens;
    pp.header = header;
    pp.part_start = part_start;
    pp.units = units;
    pp.num_seqs = a.num_seqs;
    pp.num_kv_heads = a.num_kv_heads;
    pp.q_len = a.q_len;
    pp.partition = a.partition;
    pp.max_blocks_per_seq = a.max_blocks_per_seq;
    pp.max_context_len = a.max_context_len;
    const cudaError_t pe = prefix ? launch_pdl(plan_prefix_kernel, dim3(1), dim3(1024), 0, stream, pp, *a.groups)
                                  : launch_pdl(plan_kernel, dim3(1), dim3(1024), 0, stream, pp);
    if (pe != cudaSuccess) return PA_ERR_CUDA;
    *launches += 1;
    profile_mark(pc, 1, stream);
    DecodeParams p;
    if (a.fp8) {
        if (D != 128) return PA_ERR_UNSUPPORTED;
        if (int st = make_kv_map_fp8(&p.tmap_k, a.key_cache, a.num_blocks, a.num_kv_heads, D)) return st;
        if (int st = make_kv_map_fp8(&p.tmap_v, a.value_cache, a.num_blocks, a.num_kv_heads, D)) return st;
    } else {
        if (int st = make_kv_map(&p.tmap_k, a.key_cache, a.dtype, a.num_blocks, a.num_kv_heads, D)) return st;
        if (int st = make_kv_map(&p.tmap_v, a.value_cache, a.dtype, a.num_blocks, a.num_kv_heads, D)) return st;
    }
    p.out = a.out;
    p.query = a.query;
    p.block_tables = a.block_tables;
    p.header = header;
    p.work_counter = header + 1;
    p.units = units;
    p.pml = pml;
    p.pacc = pacc;
    p.num_blocks = a.num_blocks;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.q_len = a.q_len;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.group = a.num_heads / a.num_kv_heads;
    p.total_rows = p.group * a.q_len;
    // More than 64 query rows per kv head (a prefill chunk): units take 64-row groups.
    p.rows = std::min(PA_ROW_GROUP_ROWS, p.total_rows);
    p.row_groups = (p.total_rows + p.rows - 1) / p.rows;
    p.partition = a.partition;
    p.scale_log2 = a.scale * (a.fp8 ? a.k_scale : 1.f) * 1.4426950408889634f;
    p.v_scale = a.fp8 ? a.v_scale : 1.f;
    p.wait_limit_ns = static_cast<unsigned int>(wait_limit_ns());
    // Each consumer warp owns 8 (NT = 1) or 16 (NT = 2) query rows of the kv head; the row
    // tiles per kv head are rounded up to a divisor of the consumer warp count (a third
    // tile becomes a fourth, all-padding one) so that every consumer warp owns exactly one
    // (row tile, block split) pair.
    int rt, nt;
    decode_variant(p.rows, a.fp8, rt, nt);
    const int tile_rows = 8 * nt;
    p.mtiles = (p.rows + tile_rows - 1) / tile_rows;
    if (p.mtiles == 3) p.mtiles = 4;
    if (p.mtiles > kConsumerWarps || kConsumerWarps % p.mtiles != 0) return PA_ERR_UNSUPPORTED;
    p.block_splits = kConsumerWarps / p.mtiles;
    p.slot_rows = std::min(tile_rows, p.rows);

    using KernelFn = void (*)(DecodeParams);
    KernelFn kfn;
    if constexpr (D == 128) {
        if (a.fp8) kfn = nt == 1 ? decode_kernel<T, D, 1, 0, true> : decode_kernel<T, D, 2, 0, true>;
    }
    if (!a.fp8)
        kfn = rt == 1   ? decode_kernel<T, D, 1, 1, false>
              : rt == 2 ? decode_kernel<T, D, 1, 2, false>
              : rt == 4 ? decode_kernel<T, D, 1, 4, false>
              : rt == 8 ? decode_kernel<T, D, 1, 8, false>
              : nt == 1 ? decode_kernel<T, D, 1, 0, false>
                        : decode_kernel<T, D, 2, 0, false>;
    const void* fn = reinterpret_cast<const void*>(kfn);
    const int ctas_target = decode_ctas_per_sm(nt, rt, a.fp8);
    // Deepest ring that still lets ctas_target CTAs share an SM.  Its length must be a
    // multiple of block_splits: then every stage is always consumed by the same warps,
    // which wait its phases strictly in order (a waiter two phases ahead of a barrier
    // would see its parity as already complete).
    int stages = (kMaxStages / p.block_splits) * p.block_splits;
    if (stages < p.block_splits) return PA_ERR_UNSUPPORTED;
    SmemLayout lay = smem_layout(D, stages, p.mtiles, tile_rows, p.slot_rows, rt > 0, a.fp8);
    const int per_sm_budget = 228 * 1024 / ctas_target - 1024;
    while (stages > p.block_splits && lay.total > per_sm_budget) {
        stages -= p.block_splits;
        lay = smem_layout(D, stages, p.mtiles, tile_rows, p.slot_rows, rt > 0, a.fp8);
    }
    if (lay.total > dev.max_smem_optin) return PA_ERR_UNSUPPORTED;
    p.stages = stages;
    int per_sm = 1;
    if (int st = decode_blocks_per_sm(fn, lay.total, per_sm)) return st;
    const long long max_units = (long long)a.num_seqs * w.pmax * a.num_kv_heads * p.row_groups;
    const int grid = (int)std::max(1LL, std::min<long long>((long long)dev.sms * per_sm, max_units));

    const cudaError_t le = launch_pdl(kfn, dim3(grid), dim3(kThreads), lay.total, stream, p);
    if (le != cudaSuccess) return PA_ERR_CUDA;
    profile_mark(pc, 2, stream);
    *launches += 1;
    // Shared prefixes: one tcgen05 pass per (group, kv head) over every grouped row, after the
    // partition pass under programmatic launch.  Its CTAs (one per SM) take the SMs the partition
    // pass's CTAs leave as they run out of work, and its epilogue, once the partition pass has
    // finished, merges every grouped sequence's pieces and writes the output rows.
    bool merge_needed = w.pmax > 1;
    if (prefix) {
        if (int st = launch_prefix_tc(a, part_start, pml, pacc, stream, launches)) return st;
        // Only sequences outside every group with a prefix can still be split.
        const PrefixGroups& g = *a.groups;
        int covered = 0;
        for (int k = 0; k < g.n; ++k)
            if (g.len[k] > 0) covered += g.seq_start[k + 1] - g.seq_start[k];
        merge_needed = covered < a.num_seqs;
    }

    if (merge_needed) {
        MergeParams mp;
        mp.out = a.out;
        mp.part_start = part_start;
        mp.pml = pml;
        mp.pacc = pacc;
        mp.num_seqs = a.num_seqs;
        mp.q_len = a.q_len;
        mp.num_heads = a.num_heads;
        const long long rows = (long long)a.num_seqs * a.q_len * a.num_heads;
        const unsigned blocks = (unsigned)((rows * 32 + 127) / 128);
        const cudaError_t me = prefix
                                   ? launch_pdl(merge_ungrouped_kernel<T, D>, dim3(blocks), dim3(128), 0, stream, mp,
                                                *a.groups)
                                   : launch_pdl(merge_kernel<T, D>, dim3(blocks), dim3(128), 0, stream, mp);
        if (me != cudaSuccess) return PA_ERR_CUDA;
        *launches += 1;
    }
    profile_mark(pc, 3, stream);
    return PA_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// Pieces shared with the other kernel translation units (pa_internal.h).
// ---------------------------------------------------------------------------
int kv_tensor_map(CUtensorMap* map, const void* base, int dtype, int64_t num_blocks, int num_kv_heads,
                  int head_dim) {
    return make_kv_map(map, base, dtype, num_blocks, num_kv_heads, head_dim);
}

int device_error_word(int** ptr) {
    static int* cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!cached[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_error) != cudaSuccess || !p) return PA_ERR_CUDA;
        cached[dev] = static_cast<int*>(p);
    }
    *ptr = cached[dev];
    return PA_OK;
}

int sm_count(int* sms) {
    DeviceInfo d;
    if (int st = device_info(d)) return st;
    *sms = d.sms;
    return PA_OK;
}

int ensure_dynamic_smem(const void* fn, int smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    DeviceInfo d;
    if (int st = device_info(d)) return st;
    if (smem > d.max_smem_optin) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return PA_ERR_CUDA;
    // Raised to what this call needs and never lowered.
    if (fa.maxDynamicSharedSizeBytes < smem &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

int profile_call_begin() {
    if (!g_prof.mode || g_prof.n >= kProfCalls) return -1;
    return g_prof.n++;
}

void profile_mark(int call, int mark, cudaStream_t stream) {
    if (call < 0 || (mark == 2 && g_prof.mode == 2)) return;
    cudaEventRecord(g_prof.ev[4 * call + mark], stream);
}

int launch_reshape_and_cache(const void* key, const void* value, void* key_cache, void* value_cache,
                             const int64_t* slot_mapping, int64_t num_tokens, int row_bytes,
                             int64_t num_slots, cudaStream_t stream, int* launches) {
    DeviceInfo dev;
    if (int st = device_info(dev)) return st;
    const int row_vecs = row_bytes / 16;
    const long long total = (long long)num_tokens * 2 * row_vecs;
    const long long want = (total + 255) / 256;
    const int grid = (int)std::max(1LL, std::min<long long>(want, (long long)dev.sms * 8));
    if (launch_pdl(reshape_kernel, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(key),
                   static_cast<const uint4*>(value), static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache),
                   reinterpret_cast<const long long*>(slot_mapping), (long long)num_tokens, row_vecs,
                   (long long)num_slots) != cudaSuccess)
        return PA_ERR_CUDA;
    *launches += 1;
    return PA_OK;
}

int launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache, void* value_cache,
                                 const int64_t* slot_mapping, int64_t num_tokens, int row_elems, int64_t num_slots,
                                 int dtype, float k_scale, float v_scale, cudaStream_t stream, int* launches) {
    DeviceInfo dev;
    if (int st = device_info(dev)) return st;
    const int row_vecs = row_elems / 8;
    const long long total = (long long)num_tokens * 2 * row_vecs;
    const int grid = (int)std::max(1LL, std::min<long long>((total + 255) / 256, (long long)dev.sms * 8));
    const auto* k = static_cast<const uint4*>(key);
    const auto* v = static_cast<const uint4*>(value);
    auto* kc = static_cast<uint2*>(key_cache);
    auto* vc = static_cast<uint2*>(value_cache);
    const auto* sm = reinterpret_cast<const long long*>(slot_mapping);
    const cudaError_t le =
        dtype == PA_BF16 ? launch_pdl(reshape_fp8_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, k, v, kc, vc,
                                      sm, (long long)num_tokens, row_vecs, (long long)num_slots, k_scale, v_scale)
                         : launch_pdl(reshape_fp8_kernel<__half>, dim3(grid), dim3(256), 0, stream, k, v, kc, vc, sm,
                                      (long long)num_tokens, row_vecs, (long long)num_slots, k_scale, v_scale);
    if (le != cudaSuccess) return PA_ERR_CUDA;
    *launches += 1;
    return PA_OK;
}

int launch_copy_blocks(void* key_cache, void* value_cache, const int64_t* block_mapping, int64_t num_pairs,
                       int block_bytes, int64_t num_blocks, cudaStream_t stream, int* launches) {
    DeviceInfo dev;
    if (int st = device_info(dev)) return st;
    const int block_vecs = block_bytes / 16;
    const long long total = (long long)num_pairs * 2 * block_vecs;
    const long long want = (total + 255) / 256;
    const int grid = (int)std::max(1LL, std::min<long long>(want, (long long)dev.sms * 16));
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache),
                                                 reinterpret_cast<const long long*>(block_mapping), num_pairs,
                                                 block_vecs, num_blocks);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    *launches += 1;
    return PA_OK;
}

int launch_spec_verify(int32_t* num_accepted, int32_t* out_tokens, const float* target_probs,
                       const float* draft_probs, const int32_t* draft_tokens, const float* u_accept,
                       const float* u_sample, int num_seqs, int k, int vocab, cudaStream_t stream, int* launches) {
    SpecParams p;
    p.num_accepted = num_accepted;
    p.out_tokens = out_tokens;
    p.target = target_probs;
    p.draft = draft_probs;
    p.draft_tokens = draft_tokens;
    p.u_accept = u_accept;
    p.u_sample = u_sample;
    p.k = k;
    p.vocab = vocab;
    // One cluster of kSpecCluster CTAs per sequence.
    if (num_seqs > 0x7fffffff / kSpecCluster) return PA_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_seqs * kSpecCluster);
    cfg.blockDim = dim3(kSpecThreads);
    if (int st = ensure_dynamic_smem(reinterpret_cast<const void*>(spec_verify_kernel), kSpecStageBytes)) return st;
    cfg.dynamicSmemBytes = kSpecStageBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSpecCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, spec_verify_kernel, p) != cudaSuccess) return PA_ERR_CUDA;
    *launches += 1;
    return PA_OK;
}

// Prefill chunks (many query rows per kv head) run on the tcgen05 kernel: in auto mode
// when a kv head has at least PA_TC_MIN_ROWS query rows and the caller left the split to
// the library, and always in tcgen05 mode (16-bit caches).
bool use_prefill_tc(const DecodeArgs& a) {
    if (a.fp8) return false;
    if (g_decode_math == 3) return true;
    const long long rows = (long long)(a.num_heads / a.num_kv_heads) * a.q_len;
    return g_decode_math == 0 && a.partition_auto && rows >= PA_TC_MIN_ROWS;
}

int launch_decode(const DecodeArgs& args, cudaStream_t stream, int* launches, int* partition_used) {
    *partition_used = 0;
    if (!args.groups && use_prefill_tc(args)) return launch_prefill_tc(args, stream, launches);  // no split
    if (args.groups && !args.fp8 && (args.num_heads / args.num_kv_heads) * args.q_len >= kTcSuffixMinRows) {
        // Shared prefixes with enough rows per kv head: suffixes and prefixes on tcgen05 (no split;
        // the suffix pieces go to the workspace's first per-sequence partial slots).
        const WsLayout w = ws_layout(args.num_seqs, args.q_len, args.num_heads, args.head_dim, args.max_context_len,
                                     args.partition, true);
        uint8_t* ws = static_cast<uint8_t*>(args.workspace);
        return launch_shared_prefix_tc(args, reinterpret_cast<float2*>(ws + w.pml), reinterpret_cast<float*>(ws + w.pacc),
                                       reinterpret_cast<int*>(ws + w.order), stream, launches);
    }
    DecodeArgs a = args;
    if (a.partition_auto) {
        DeviceInfo dev;
        if (int st = device_info(dev)) return st;
        // >= the partition the workspace was sized for (the default, or the smallest prefix one)
        a.partition = a.groups ? auto_partition_prefix(a, dev.sms) : auto_partition(a, dev.sms);
    }
    *partition_used = a.partition;
    if (a.dtype == PA_BF16) {
        if (a.head_dim == 128) return launch_decode_typed<__nv_bfloat16, 128>(a, stream, launches);
        if (a.head_dim == 64) return launch_decode_typed<__nv_bfloat16, 64>(a, stream, launches);
    } else {
        if (a.head_dim == 128) return launch_decode_typed<__half, 128>(a, stream, launches);
        if (a.head_dim == 64) return launch_decode_typed<__half, 64>(a, stream, launches);
    }
    return PA_ERR_UNSUPPORTED;
}

int read_device_error(int32_t* flags, int clear, cudaStream_t stream) {
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_pa_error, sizeof(int), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_pa_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return PA_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
    }
    *flags = v;
    return PA_OK;
}

// Limit of the kernels' pipeline waits, copied into every launch's parameters.
std::atomic<unsigned long long> g_wait_limit_ns{kWaitLimitNs};

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int set_wait_limit_ns(unsigned long long ns) {
    g_wait_limit_ns.store(ns == 0 || ns > kWaitLimitNs ? kWaitLimitNs : ns, std::memory_order_relaxed);
    return PA_OK;
}

int set_decode_math(int math) {
    if (math < 0 || math > 3) return PA_ERR_INVALID_ARG;
    g_decode_math = math;
    return PA_OK;
}

int profile_enable(int on) {
    if (on < 0 || on > 2) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    if (on && !g_prof.created) {
        for (int i = 0; i < 4 * kProfCalls; ++i)
            if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) return PA_ERR_CUDA;
        g_prof.created = true;
        cudaGetDevice(&g_prof.dev);
    }
    if (on != g_prof.mode) g_prof.n = 0;  // a record never mixes modes
    g_prof.mode = on;
    return PA_OK;
}

int profile_read_parts(float* plan_ms, float* main_ms, float* merge_ms, int* calls) {
    std::lock_guard<std::mutex> lk(g_mu);
    float sum[3] = {0.f, 0.f, 0.f};
    for (int i = 0; i < g_prof.n; ++i) {
        const cudaEvent_t* e = g_prof.ev + 4 * i;
        if (cudaEventSynchronize(e[3]) != cudaSuccess) return PA_ERR_CUDA;
        float ms[3] = {0.f, 0.f, 0.f};
        if (cudaEventElapsedTime(&ms[0], e[0], e[1]) != cudaSuccess) return PA_ERR_CUDA;
        if (g_prof.mode == 2) {
            if (cudaEventElapsedTime(&ms[1], e[1], e[3]) != cudaSuccess) return PA_ERR_CUDA;
        } else {
            if (cudaEventElapsedTime(&ms[1], e[1], e[2]) != cudaSuccess) return PA_ERR_CUDA;
            if (cudaEventElapsedTime(&ms[2], e[2], e[3]) != cudaSuccess) return PA_ERR_CUDA;
        }
        for (int k = 0; k < 3; ++k) sum[k] += ms[k];
    }
    *plan_ms = sum[0];
    *main_ms = sum[1];
    *merge_ms = sum[2];
    *calls = g_prof.n;
    g_prof.n = 0;
    return PA_OK;
}

// ---------------------------------------------------------------------------
// Fixed scratch for pa_decode_attention_noalloc.
//
// Callers that must not allocate device memory get their split-K workspace from
// this array instead of passing one in.  It is a module global: every GPU that
// loads the library holds PA_NOALLOC_WORKSPACE_BYTES of it until the process
// exits.  In host code `g_noalloc_workspace` only names the array; its device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and cached.  All calls share the array and it keeps the last
// call's contents; the decode kernels rewrite every byte they read from it on
// each call (work list, partials), so nothing needs clearing between calls.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_workspace[PA_NOALLOC_WORKSPACE_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};
}  // namespace

int noalloc_workspace(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return PA_OK;
}

}  // namespace pa
