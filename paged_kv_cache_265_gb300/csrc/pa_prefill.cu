// pa_prefill.cu -- attention of prefill chunks over the paged KV cache on the
// fifth-generation tensor cores: tcgen05.mma with its accumulators and the
// softmax weights in tensor memory (TMEM), K/V blocks staged in shared memory by
// tensor-map TMA.
//
// It computes exactly what the multi-query decode path computes: the q_len
// chunk tokens are the last q_len positions of each sequence, and query row j
// sees positions 0 .. L - q_len + j ("现代 LLM 推理引擎剖析", section 2.1 Chunked
// Prefill: a long prompt is run in chunks, each attending to the cache its
// earlier chunks filled; the attention is the dense causal definition of "LLM
// 推理优化的系统视角", section 3.1, with the query-head grouping of its section
// 3.2).  A chunk has g * q_len query rows per kv head, enough to fill 128-row
// tensor-core tiles, so the context is not split.
//
// One CTA = one tile of 128 query rows of one kv head.  Rows are token-major
// (row r of a kv head is chunk token r / g, query head kvh * g + r % g), so a
// tile spans 128 / g consecutive chunk tokens whose causal limits are close.
// For each K/V tile j of 128 positions (8 pool blocks):
//   S_j = Q K^T   M = 128, N = 16 x blocks, K = D: A = Q, held in TMEM for the
//                 whole CTA (columns 384 .. 384 + D/2 - 1, two elements per
//                 column), B = K tile from shared memory (K-major, 128-byte
//                 swizzled); S_j (fp32) into TMEM buffer j % 2 (columns 0-127 or
//                 128-255).  With both operands in shared memory a 128 x 128
//                 product is limited by the shared-memory operand reads; with A
//                 in TMEM it runs at the tensor rate
//   softmax       warps 0-7: warps w and w + 4 share TMEM lanes 32 (w % 4) ..,
//                 so each tile row (lane) has two threads, one per 64-column
//                 half.  A thread reads the other half only for the row max,
//                 then masks, exponentiates (ex2.approx of the log2-scaled scores
//                 against a running max that is raised only when it grows by
//                 more than 8: weights stay <= 2^8 and the final division uses
//                 the same max, so only rounding changes) and writes back its own
//                 half.  Each weight p is split into p_hi = p rounded to the input
//                 type and p_lo = (p - p_hi) rounded (about 16 significant bits
//                 reach the product; one 16-bit P alone misses the attention
//                 tolerance when a few positions dominate); for positions 64 h ..
//                 64 h + 63 they go back over the same S columns, P_hi in the
//                 first 32 and P_lo in the next 32 (two weights per column)
//   O += P V      M = 128, N = D, K = 16 x blocks, A = P_hi then P_lo straight
//                 from TMEM, B = V tile (MN-major: d is contiguous in the
//                 cache); O (fp32) in TMEM columns 256 .. 256 + D - 1
// With two S buffers, S_{j+1} runs on the tensor cores while the softmax warps
// work on S_j, and P_j V_j while they start on S_{j+1}.
//
// Warps: 0-7 softmax and epilogue, 8 TMA producer (K/V blocks found through the
// block table, three stages of one K/V tile), 9 TMEM owner and MMA issuer (one
// thread).  Every wait is bounded (PA_DEVERR_TIMEOUT); a failed wait stops all
// roles, and the CTA lets its copies and products finish before it frees TMEM.
//
// Shared-prefix mode (prefix_tc_kernel): sequences that map the same prefix blocks
// ("每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速", section "KV Cache 又大又碎，
// 为何不用操作系统分页的思路管它？": one physical block mapped by many sequences) see the
// same prefix K/V, so one CTA takes 128 query rows of several sequences of a group (row r =
// sequence r / (g q_len), then chunk token, then head) against the whole prefix, with no
// causal mask (every chunk row lies after the prefix).  It is launched after the split-K
// partition pass has covered the rest of each sequence; its epilogue merges the prefix piece
// with those pieces by their log-sum-exp and writes the output rows.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

#ifndef PA_TC_SUFFIX_PERSISTENT
#define PA_TC_SUFFIX_PERSISTENT 1
#endif
// Kernel modes whose softmax takes its weights in packed fp32 pairs (bit m: mode m): fewer
// instructions shorten the chain of the suffix kernel's few-row tiles, while beside eight busy
// softmax warps (full tiles) the denser arithmetic slows the tensor-core products.
#ifndef PA_TC_PACKED_MODES
#define PA_TC_PACKED_MODES 4
#endif

constexpr int kTcRows = 128;             // query rows per CTA tile (MMA M)
constexpr int kTcPos = 128;              // positions per K/V tile
constexpr int kTcBlocks = kTcPos / 16;   // pool blocks per K/V tile
constexpr int kTcStages = 3;             // K/V tiles in flight
constexpr int kTcThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;           // S / P buffers: columns 0-127 and 128-255
constexpr uint32_t kTmemO = 256;         // O columns
constexpr uint32_t kTmemQ = 384;         // Q: two 16-bit elements per column
constexpr int kRegion = kTcRows * 128;   // 128 rows x 128 B: one 64-element column block
constexpr int kBox = 16 * 128;           // one TMA box: 16 positions x 64 elements

struct PrefillTcParams {
    CUtensorMap tmap_k;  // 64-byte aligned members first
    CUtensorMap tmap_v;
    void* out;
    const void* query;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int* err;
    int max_blocks_per_seq;
    int num_blocks;
    int q_len;
    int num_heads;
    int num_kv_heads;
    int group;       // query heads per kv head
    int total_rows;  // group * q_len query rows per kv head
    int mtiles;      // 128-row tiles per kv head
    int max_context_len;
    int num_units;   // chunk and suffix modes: (sequence, kv head, 128-row tile) units
    float scale_log2;
    unsigned int wait_limit_ns;  // limit of the pipeline waits (pa_set_wait_limit_ns), at most 2 s
    // Shared-prefix mode: the other pieces of each sequence, merged with the prefix's.
    const int* part_start;  // first partial slot of each sequence (the prefix piece's, not stored)
    const float2* pml;      // (max in log2 units, sum) per partial row
    const float* pacc;      // unnormalised partial outputs, fp32
    // Suffix mode: where a sequence with a shared prefix leaves its suffix piece (slot i).
    float2* pml_out;
    float* pacc_out;
    // Suffix mode: the units, longest first (null: index order).
    const int* order;
};

template <int D>
struct TcLayout {
    static constexpr int kHalves = D / 64;                 // 64-element column blocks of d
    static constexpr int kStage0 = 0;                      // stages: K tile then V tile
    static constexpr int kKBytes = kHalves * kRegion;
    static constexpr int kStageBytes = 2 * kKBytes;
    static constexpr int kBars = kStage0 + kTcStages * kStageBytes;
    // barriers (8 B each): kvfull[3] +0, kvempty[3] +24, sfull[2] +48, pfull +64, odone +72,
    // drain +80, qready +88, lready +96; TMEM base +104; abort flag +108; the two half-row
    // sums of every row at +128 (float [2][128])
    static constexpr int kTotal = kBars + 128 + 1024;
    static constexpr int kAlloc = kTotal + 1024;           // slack to align the base to 1024 B
};

__device__ __forceinline__ float lo16(uint32_t v, std::true_type /*bf16*/) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float hi16(uint32_t v, std::true_type) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float lo16(uint32_t v, std::false_type /*fp16*/) {
    return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu)));
}
__device__ __forceinline__ float hi16(uint32_t v, std::false_type) {
    return __half2float(__ushort_as_half((unsigned short)(v >> 16)));
}

// max(a, b, c) in one instruction (the softmax's row maxima are most of its non-exponential work).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed pairs of fp32 (one 64-bit register, two lanes of arithmetic per instruction): each lane
// rounds as the scalar instruction does.
__device__ __forceinline__ unsigned long long f2_make(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Bits of the columns in [lo, hi] that fall in the 32-column word starting at `base`.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int base) {
    const int a = max(lo - base, 0), b = min(hi - base, 31);
    if (b < a) return 0u;
    const uint32_t upto_b = b == 31 ? 0xffffffffu : ((1u << (b + 1)) - 1u);
    return upto_b & ~((1u << a) - 1u);
}

// D[tmem] (+)= A[tmem] * B[smem] (kAccumulate: add to D, else overwrite it), issued by one
// thread: the A operand (M = 128 rows in TMEM lanes, two 16-bit K elements per column, the
// even one in the low half) is read from tensor memory.
template <bool kAccumulate>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "n"(kAccumulate ? 1 : 0)
        : "memory");
}

// The tile's sequence, rows and positions.  Chunk mode: one sequence's q_len chunk rows of one
// kv head against its positions 0 .. L - 1 under the causal limits.  Prefix mode: rows of every
// sequence of one prefix group (row r = sequence r / (g q_len), chunk token, head) against the
// group's shared prefix, which every row sees whole.
struct TcTile {
    int seq;       // the sequence whose block table the tile walks (prefix mode: the group's first)
    int kvh;
    int row0;      // first row of the tile among the kv head's rows
    int rows;      // rows of the kv head (past them a tile row is padding)
    int L;         // chunk mode: the sequence's length; prefix mode: the prefix length
    bool valid;
    int nblk;      // pool blocks the tile streams
    int lastblk;   // the last of them (counted from blk0) is short by sh rows (chunk modes only)
    int sh;
    int blk0;      // first pool block of the tile's positions, in the sequence's table
};

// Kernel modes: the chunk kernel, the shared-prefix kernel, and the suffix kernel (chunk rows
// against the positions after each sequence's shared prefix).
enum : int { kModeChunk = 0, kModePrefix = 1, kModeSuffix = 2 };

template <int kMode>
__device__ __forceinline__ TcTile tc_tile(const PrefillTcParams& p, const PrefixGroups* g, int idx) {
    constexpr bool kPrefix = kMode == kModePrefix;
    TcTile w;
    if constexpr (kPrefix) {
        int lo = 0, hi = g->n - 1;  // the group whose tiles hold this unit
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (g->tile_start[mid] <= idx) lo = mid; else hi = mid - 1;
        }
        w.seq = g->seq_start[lo];
        w.rows = (g->seq_start[lo + 1] - w.seq) * p.total_rows;
        const int mtiles = (w.rows + kTcRows - 1) / kTcRows;
        const int local = idx - g->tile_start[lo];
        w.row0 = (local % mtiles) * kTcRows;
        w.kvh = local / mtiles;
        w.L = g->len[lo];
        w.valid = w.L > 0;
        w.nblk = w.L / 16;
        w.lastblk = w.nblk - 1;
        w.sh = 0;
        w.blk0 = 0;
    } else {
        // Tiles of one (sequence, kv head) are adjacent and share its K/V in L2; the
        // last rows (the longest causal ranges) go first.
        const int mt = p.mtiles - 1 - idx % p.mtiles;
        w.kvh = (idx / p.mtiles) % p.num_kv_heads;
        w.seq = idx / (p.mtiles * p.num_kv_heads);
        w.row0 = mt * kTcRows;
        w.rows = p.total_rows;
        w.L = p.context_lens[w.seq];
        // Suffix mode: the positions before the sequence's shared prefix end are another kernel's.
        const int skip = kMode == kModeSuffix ? prefix_of(*g, w.seq) : 0;
        w.blk0 = skip / 16;
        w.valid = seq_len_valid(w.L, p.q_len, skip, p.max_context_len, p.max_blocks_per_seq);
        const int t_last = min((w.row0 + kTcRows - 1) / p.group, p.q_len - 1);
        // blocks this tile sees, counted from block blk0
        w.nblk = w.valid ? (w.L - p.q_len + t_last) / 16 + 1 - w.blk0 : 0;
        w.lastblk = (w.L - 1) / 16 - w.blk0;      // the sequence's last block ...
        w.sh = 16 * ((w.L - 1) / 16 + 1) - w.L;   // ... is short by sh rows, fetched as leading zeros
    }
    return w;
}

// The k-th unit this CTA takes, or -1 when it has no more.  With an order (suffix mode, units
// sorted longest first) the CTAs take its positions back and forth, CTA b positions b,
// 2G - 1 - b, 2G + b, ... of G CTAs, which balances their sums of unit lengths; otherwise
// units b, b + G, ... (one unit per CTA in chunk mode, where G is the unit count).
__device__ __forceinline__ int tc_unit(const PrefillTcParams& p, int num_units, int k) {
    const int G = (int)gridDim.x, b = (int)blockIdx.x;
    if (p.order) {
        const long long pos = (long long)k * G + ((k & 1) ? G - 1 - b : b);
        return pos < num_units ? __ldg(p.order + pos) : -1;
    }
    const long long u = (long long)k * G + b;
    return u < num_units ? (int)u : -1;
}

template <typename T, int D, int kMode>
__device__ __forceinline__ void tc_attention(const PrefillTcParams& p, const PrefixGroups* g) {
    constexpr bool kPrefix = kMode == kModePrefix;
    using Lay = TcLayout<D>;
    using IsBf16 = std::integral_constant<bool, std::is_same<T, __nv_bfloat16>::value>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t st_s = sbase + Lay::kStage0;
    const uint32_t bars = sbase + Lay::kBars;
    const uint32_t kvfull = bars, kvempty = bars + 24, sfull = bars + 48, pfull = bars + 64, odone = bars + 72,
                   drain = bars + 80, qready = bars + 88, lready = bars + 96;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Lay::kBars + 104);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lay::kBars + 108);
    float* lsum = reinterpret_cast<float*>(smem + Lay::kBars + 128);
    int* err = p.err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(kvfull + 8 * s, 1);
            mbar_init(kvempty + 8 * s, 1);
        }
        mbar_init(sfull, 1);
        mbar_init(sfull + 8, 1);
        mbar_init(pfull, 2 * kTcRows);
        mbar_init(odone, 1);
        mbar_init(drain, 1);
        mbar_init(qready, 2 * kTcRows);
        mbar_init(lready, 2 * kTcRows);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tc::alloc(bars + 104, kTmemCols);
        tc::relinquish_alloc_permit();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    griddep_launch_dependents();
    // Chunk mode: the appended K/V rows and the query come from earlier kernels.  Prefix mode
    // reads only the shared prefix (never appended to by this step) until its epilogue, which
    // waits for the plan kernel's partial slots.
    if constexpr (!kPrefix) griddep_wait();

    // The CTA takes the units tc_unit() names (one CTA per SM).  Every role
    // walks the same units and counts their K/V tiles in one running index gt, so stage, S
    // buffer and barrier phases carry on from one unit to the next; per-unit barriers (qready,
    // lready) count valid units (vu).  Tensor memory and the barriers are set up once.
    const int num_units = kPrefix ? g->tile_start[g->n] : p.num_units;
    // Chunk mode launches one CTA per unit: its running indices are the compile-time 0 of a
    // single unit (the loop below runs once), and the loop costs it nothing.
    constexpr bool kLoop = kMode != kModeChunk;
    const int k_end = kLoop ? 0x7fffffff : 1;

    if (warp == 8) {
        // ===================== TMA producer =====================
        int armed[kTcStages] = {0, 0, 0};
        int gt_run = 0;
        bool ok = true;
        for (int k = 0; ok && k < k_end; ++k) {
        const int u = tc_unit(p, num_units, k);
        if (u < 0) break;
        const TcTile tile = tc_tile<kMode>(p, g, u);
        if (!tile.valid) {
            if (!kPrefix && lane == 0) atomicOr(err, PA_DEVERR_CONTEXT);  // rows left untouched
            continue;
        }
        const int kvh = tile.kvh, nblk = tile.nblk, lastblk = tile.lastblk, sh = tile.sh;
        const int ntiles = (nblk + kTcBlocks - 1) / kTcBlocks;
        const int* bt = p.block_tables + (long long)tile.seq * p.max_blocks_per_seq + tile.blk0;
        // Block ids arrive 32 at a time (four tiles): lane l holds the id of block 32c + l
        // of chunk c, and chunk c + 1 is requested when chunk c starts, so no tile waits on
        // a block-table load.
        int ids = lane < nblk ? __ldg(bt + lane) : 0;
        int ids_next = 32 + lane < nblk ? __ldg(bt + 32 + lane) : 0;
        const int gtb = kLoop ? gt_run : 0;
        for (int j = 0; j < ntiles; ++j) {
            const int gt = gtb + j;
            const int s = gt % kTcStages;
            const int jj = j & 3;
            if (jj == 0 && j > 0) {
                ids = ids_next;
                const int nxt = 32 * ((j >> 2) + 1) + lane;
                ids_next = nxt < nblk ? __ldg(bt + nxt) : 0;
            }
            if (gt >= kTcStages) {
                bool w = true;
                if (lane == 0) w = mbar_wait(kvempty + 8 * s, ((gt / kTcStages) - 1) & 1, err, abort_flag, p.wait_limit_ns);
                if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
                    ok = false;
                    break;
                }
            }
            const int nb = min(kTcBlocks, nblk - kTcBlocks * j);
            const int bid = __shfl_sync(0xffffffffu, ids, (8 * jj + lane) & 31);
            const bool good = lane < nb && bid >= 0 && bid < p.num_blocks;
            if (lane < nb && !good) atomicOr(err, PA_DEVERR_BLOCK_ID);  // skipped: the tile computes on stale data
            const unsigned gm = __ballot_sync(0xffffffffu, good);
            const uint32_t bar = kvfull + 8 * s;
            if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(gm) * 2u * Lay::kHalves * kBox);
            __syncwarp();
            if (good) {
                const int y0 = (kTcBlocks * j + lane == lastblk) ? -sh : 0;  // rows before 0 arrive as zeros
                const uint32_t kdst = st_s + s * Lay::kStageBytes + lane * kBox;
#pragma unroll
                for (int h = 0; h < Lay::kHalves; ++h) {
                    tc::tma_load_4d(kdst + h * kRegion, &p.tmap_k, h * 64, kvh, y0, bid, bar);
                    tc::tma_load_4d(kdst + Lay::kKBytes + h * kRegion, &p.tmap_v, h * 64, kvh, y0, bid, bar);
                }
            }
            ++armed[s];
        }
        gt_run += ntiles;
        }
        // No copy may still be landing when the CTA exits.
        if (lane == 0)
            for (int s = 0; s < kTcStages; ++s)
                if (armed[s] > 0) mbar_wait(kvfull + 8 * s, (armed[s] - 1) & 1, err, nullptr);
        __syncwarp();
    } else if (warp == 9) {
        // ===================== MMA issuer =====================
        // Order: S_j, then P_{j-1} V_{j-1}.  S_j overwrites the buffer P_{j-2} was read
        // from, so it waits for P_{j-2} V_{j-2} to complete.
        // The tensor cores take 64 cycles per 128 x 128 x 16 product, so the issuing thread does
        // little else: descriptors are formed once per stage and each product adds a constant.
        if (lane == 0) {
            constexpr bool kBf16 = IsBf16::value;
            constexpr uint32_t id_o = tc::idesc_f16(kBf16, true, kTcRows, D);
            // Stage s adds s * kStageBytes / 16 to the start-address field of stage 0's
            // descriptors and a product's K slice its byte offset / 16; addresses stay below
            // 256 KB, so the 14-bit field never carries into the next one.
            const uint64_t kdesc0 = tc::smem_desc_sw128(st_s, 16, 1024);
            const uint64_t vdesc0 = tc::smem_desc_sw128(st_s + Lay::kKBytes, kRegion, 1024);
            bool ok = true;
            int gt_run = 0, vu_run = 0;
            for (int k = 0; ok && k < k_end; ++k) {
            const int u = tc_unit(p, num_units, k);
            if (u < 0) break;
            const TcTile tile = tc_tile<kMode>(p, g, u);
            if (!tile.valid) continue;
            const int nblk = tile.nblk;
            const int ntiles = (nblk + kTcBlocks - 1) / kTcBlocks;
            const int gt = kLoop ? gt_run : 0, vu = kLoop ? vu_run : 0;
            // The unit's Q rows are in tensor memory (and, as every softmax thread arrives only
            // after its epilogue of the previous unit, that unit's O has been read out).
            ok = mbar_wait(qready, vu & 1, err, abort_flag, p.wait_limit_ns);
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {
                    const int g1 = gt + j, s = g1 % kTcStages;
                    // S_g1 overwrites the buffer P_{g1-2} was read from.  Inside a unit the last
                    // product issued is P_{g1-2} V; at a unit's first tile the previous unit's last
                    // P_{g1-1} V is issued too, and the wait is on it (a parity wait is only
                    // meaningful for the last phase issued).
                    const int need = j == 0 ? g1 - 1 : g1 - 2;
                    ok = mbar_wait(kvfull + 8 * s, (g1 / kTcStages) & 1, err, abort_flag, p.wait_limit_ns) &&
                         (need < 0 || mbar_wait(odone, need & 1, err, abort_flag, p.wait_limit_ns));
                    if (!ok) break;
                    tc::fence_after_sync();
                    const int nb = min(kTcBlocks, nblk - kTcBlocks * j);
                    const uint32_t id_s = tc::idesc_f16(kBf16, false, kTcRows, 16 * nb);
                    const uint64_t kd = kdesc0 + (uint64_t)((s * Lay::kStageBytes) >> 4);
                    const uint32_t d_s = tmem + kTmemS + (uint32_t)(g1 & 1) * 128;
                    mma_ts<false>(d_s, tmem + kTmemQ, kd, id_s);
#pragma unroll
                    for (int kk = 1; kk < D / 16; ++kk)
                        mma_ts<true>(d_s, tmem + kTmemQ + kk * 8, kd + (((kk >> 2) * kRegion + (kk & 3) * 32) >> 4),
                                     id_s);
                    tc::commit(sfull + 8 * (g1 & 1));
                }
                if (j > 0) {
                    const int i = j - 1, g0 = gt + i, s = g0 % kTcStages;
                    ok = mbar_wait(pfull, g0 & 1, err, abort_flag, p.wait_limit_ns);
                    if (!ok) break;
                    tc::fence_after_sync();
                    const int nb = min(kTcBlocks, nblk - kTcBlocks * i);
                    const uint64_t vd = vdesc0 + (uint64_t)((s * Lay::kStageBytes) >> 4);
                    // K step kk = positions 16 kk .. 16 kk + 15: P_hi at column 64 (kk / 4) +
                    // 8 (kk % 4) of the buffer, P_lo 32 columns on; V rows 2048 B = 128 x 16 apart
                    const uint32_t p_t = tmem + kTmemS + (uint32_t)(g0 & 1) * 128;
                    if (i == 0)
                        mma_ts<false>(tmem + kTmemO, p_t, vd, id_o);
                    else
                        mma_ts<true>(tmem + kTmemO, p_t, vd, id_o);
                    mma_ts<true>(tmem + kTmemO, p_t + 32, vd, id_o);
#pragma unroll
                    for (int kk = 1; kk < kTcBlocks; ++kk) {
                        if (kk < nb) {
                            const uint32_t pa = p_t + 64 * (kk >> 2) + 8 * (kk & 3);
                            mma_ts<true>(tmem + kTmemO, pa, vd + kk * 128, id_o);
                            mma_ts<true>(tmem + kTmemO, pa + 32, vd + kk * 128, id_o);
                        }
                    }
                    tc::commit(kvempty + 8 * s);
                    tc::commit(odone);
                }
            }
            gt_run += ntiles;
            ++vu_run;
            }
            // No product may be in flight when TMEM is freed.
            tc::commit(drain);
            mbar_wait(drain, 0, err, nullptr);
        }
        __syncwarp();
    } else {
        // ===================== softmax and epilogue (warps 0-7) =====================
        const int hf = warp >> 2;                   // column half of the row this thread owns
        const int r = threadIdx.x & (kTcRows - 1);  // tile row = TMEM lane
        const uint32_t lane_tmem = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t o_half = lane_tmem + kTmemO + (D / 2) * hf;  // this thread's half of O
        const float c2 = p.scale_log2;
        bool ok = true;
        int gt_run = 0, vu_run = 0;
        for (int k = 0; ok && k < k_end; ++k) {
        const int u = tc_unit(p, num_units, k);
        if (u < 0) break;
        const TcTile tile = tc_tile<kMode>(p, g, u);
        if (!tile.valid) continue;
        const int gt = kLoop ? gt_run : 0, vu = kLoop ? vu_run : 0;
        const int seq = tile.seq, kvh = tile.kvh, row0 = tile.row0, L = tile.L, nblk = tile.nblk;
        const int lastblk = tile.lastblk, sh = tile.sh;
        const int ntiles = (nblk + kTcBlocks - 1) / kTcBlocks;
        const int gr = row0 + r;
        const bool real = gr < tile.rows;
        // the row's sequence, chunk token and query head (padding rows: the tile's first row)
        const int rseq = kPrefix ? seq + (real ? gr / p.total_rows : 0) : seq;
        const int rrow = kPrefix ? (real ? gr % p.total_rows : 0) : gr;
        const int t = real ? rrow / p.group : (kPrefix ? 0 : p.q_len - 1);
        const int hq = kvh * p.group + (real ? rrow - t * p.group : 0);
        // Last position this row sees, and the smallest such limit in the tile; a prefix row
        // sees the whole prefix.
        const int lim = kPrefix ? L - 1 : L - p.q_len + t;
        const int lim_min = kPrefix ? L - 1 : L - p.q_len + row0 / p.group;
        const long long row_id = ((long long)rseq * p.q_len + t) * p.num_heads + hq;
        const long long row_off = row_id * D;

        // This thread's half of the Q row into TMEM lane r (rows past the chunk are zeros):
        // 32-bit column c holds elements 2c (low half) and 2c + 1, as the row lies in memory.
        {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.query) + row_off) + hf * (D / 16);
            uint32_t qv[32];
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                const uint4 v = real ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                qv[4 * c] = v.x;
                qv[4 * c + 1] = v.y;
                qv[4 * c + 2] = v.z;
                qv[4 * c + 3] = v.w;
            }
            if constexpr (D == 128) {
                tc::st_x32(lane_tmem + kTmemQ + 32 * hf, qv);
            } else {
                uint32_t q16[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) q16[c] = qv[c];
                tc::st_x16(lane_tmem + kTmemQ + 16 * hf, q16);
            }
            tc::wait_st();
            tc::fence_before_sync();
            mbar_arrive(qready);
        }

        float m_run = -INFINITY, l_run = 0.f;
        // A warp whose 32 tile rows are all padding (a tile of a few real rows) computes nothing:
        // its weights and outputs are never used.  It still waits for each tile's scores and for
        // the previous tile's products before it arrives, so its arrivals for a tile never mix
        // with the next tile's (for a unit's first tile its epilogue of the previous unit waited).
        const bool idle = row0 + 32 * (warp & 3) >= tile.rows;
        for (int j = 0; j < ntiles; ++j) {
            const int g1 = gt + j;
            if (!__all_sync(0xffffffffu, mbar_wait(sfull + 8 * (g1 & 1), (g1 >> 1) & 1, err, abort_flag, p.wait_limit_ns))) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            if (idle) {
                if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(odone, (g1 - 1) & 1, err, abort_flag, p.wait_limit_ns))) {
                    ok = false;
                    break;
                }
                mbar_arrive(pfull);
                continue;
            }
            const uint32_t buf = lane_tmem + kTmemS + (uint32_t)(g1 & 1) * 128;
            const int nb = min(kTcBlocks, nblk - kTcBlocks * j);
            const int pos0 = 16 * tile.blk0 + kTcPos * j;
            // Column c holds position pos0 + c, except in the sequence's short last block
            // (columns lastc .. lastc + 15), whose first sh columns are zero rows and whose
            // column c holds position pos0 + c - sh.
            const bool short_here = sh > 0 && lastblk < kTcBlocks * j + nb;
            const bool edge = nb < kTcBlocks || short_here || pos0 + kTcPos - 1 > lim_min;
            // Scores go to log2 units as s * c2 - m in one FFMA per weight, on every path, so a
            // row's result does not depend on which other rows share its tile.  With a positive
            // scale the max is taken on the raw scores (masked columns become -inf); a
            // non-positive scale pre-multiplies every column instead.
            const bool raw = c2 > 0.f;
            const float cs = raw ? c2 : 1.f;
            const bool transform = edge || !raw;
            uint32_t vm[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
            if (edge) {  // visible columns: [0, hi1] and [lo2, hi2], as a 128-bit mask
                const int lastc = short_here ? 16 * (lastblk - kTcBlocks * j) : 16 * nb;
                const int hi1 = min(min(lim - pos0, 16 * nb - 1), lastc - 1);
                const int lo2 = short_here ? lastc + sh : 128;
                const int hi2 = min(lim - pos0 + sh, 16 * nb - 1);
#pragma unroll
                for (int k = 0; k < 4; ++k) vm[k] = range_bits(0, hi1, 32 * k) | range_bits(lo2, hi2, 32 * k);
            }
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
            {  // the other half of the row, for the row max only
                const int oh = hf ^ 1;
                uint32_t ov[64];
                tc::ld_x64(buf + 64 * oh, ov);
                if (transform) {
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        const uint32_t w = vm[2 * oh + (c >> 5)];
                        const float v0 = __uint_as_float(ov[c]), v1 = __uint_as_float(ov[c + 1]);
                        const float x0 = ((w >> (c & 31)) & 1u) ? (raw ? v0 : v0 * c2) : -INFINITY;
                        const float x1 = ((w >> ((c + 1) & 31)) & 1u) ? (raw ? v1 : v1 * c2) : -INFINITY;
                        mx[(c >> 1) & 7] = fmax3f(mx[(c >> 1) & 7], x0, x1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 64; c += 2)
                        mx[(c >> 1) & 7] = fmax3f(mx[(c >> 1) & 7], __uint_as_float(ov[c]), __uint_as_float(ov[c + 1]));
                }
            }
            uint32_t sv[64];
            tc::ld_x64(buf + 64 * hf, sv);
            if (transform) {
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const uint32_t w = vm[2 * hf + (c >> 5)];
                    const float v0 = __uint_as_float(sv[c]), v1 = __uint_as_float(sv[c + 1]);
                    const float x0 = ((w >> (c & 31)) & 1u) ? (raw ? v0 : v0 * c2) : -INFINITY;
                    const float x1 = ((w >> ((c + 1) & 31)) & 1u) ? (raw ? v1 : v1 * c2) : -INFINITY;
                    sv[c] = __float_as_uint(x0);
                    sv[c + 1] = __float_as_uint(x1);
                    mx[(c >> 1) & 7] = fmax3f(mx[(c >> 1) & 7], x0, x1);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 64; c += 2)
                    mx[(c >> 1) & 7] = fmax3f(mx[(c >> 1) & 7], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
            }
            float tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            if (raw) tmax *= c2;
            // Both threads of a row see the same maxima, so they take the same decisions.
            float alpha = 1.f;
            const bool bump = tmax > m_run + 8.f;
            if (bump) {
                alpha = ex2(m_run - tmax);
                m_run = tmax;
            }
            const float msub = m_run == -INFINITY ? 0.f : m_run;
            uint32_t ph[32], pl[32];  // P_hi and P_lo of positions 64 hf .., two weights per register
            float sum;
            if constexpr (((PA_TC_PACKED_MODES >> kMode) & 1) == 0) {
                float sm[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) sm[u] = 0.f;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float p0 = ex2(fmaf(__uint_as_float(sv[2 * c]), cs, -msub));
                    const float p1 = ex2(fmaf(__uint_as_float(sv[2 * c + 1]), cs, -msub));
                    ph[c] = Elem<T>::pack(p0, p1);
                    pl[c] = Elem<T>::pack(p0 - lo16(ph[c], IsBf16()), p1 - hi16(ph[c], IsBf16()));
                    sm[c & 7] += p0 + p1;
                }
                sum = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
            } else {
                // Weights two at a time in packed fp32 pairs: one FFMA, one residual subtraction and
                // one accumulation per pair.
                const unsigned long long cs2 = f2_make(cs, cs), nm2 = f2_make(-msub, -msub);
                unsigned long long sm2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x0, x1;
                    f2_split(f2_fma(f2_make(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), cs2, nm2), x0, x1);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    ph[c] = Elem<T>::pack(p0, p1);
                    const unsigned long long p2 = f2_make(p0, p1);
                    float r0, r1;
                    f2_split(f2_sub(p2, f2_make(lo16(ph[c], IsBf16()), hi16(ph[c], IsBf16()))), r0, r1);
                    pl[c] = Elem<T>::pack(r0, r1);
                    sm2[c & 3] = f2_add(sm2[c & 3], p2);
                }
                float sa, sb, sc, sd, se, sf, sg, sh;
                f2_split(sm2[0], sa, sb);
                f2_split(sm2[1], sc, sd);
                f2_split(sm2[2], se, sf);
                f2_split(sm2[3], sg, sh);
                sum = ((sa + sb) + (sc + sd)) + ((se + sf) + (sg + sh));
            }
            tc::st_x32(buf + 64 * hf, ph);
            tc::st_x32(buf + 64 * hf + 32, pl);
            // P_{j-1} V_{j-1} must be done before O is rescaled.
            if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(odone, (g1 - 1) & 1, err, abort_flag, p.wait_limit_ns))) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            if (j > 0 && __any_sync(0xffffffffu, bump)) {
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    uint32_t o[32];
                    tc::ld_x32(o_half + 32 * h, o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tc::st_x32(o_half + 32 * h, o);
                }
            }
            tc::wait_st();
            l_run = l_run * alpha + sum;
            tc::fence_before_sync();
            mbar_arrive(pfull);
        }
        // A wait that gave up above may have left this thread's P stores in flight: they
        // complete before tensor memory is freed.
        tc::wait_st();

        // Epilogue: the row's two half sums, then O / l, rounded once, to out[seq, t, hq, :]
        // (this thread's half of the columns); in prefix mode merged first with the sequence's
        // other pieces.
        if (ok && __all_sync(0xffffffffu, mbar_wait(odone, (gt + ntiles - 1) & 1, err, abort_flag, p.wait_limit_ns))) {
            lsum[hf * kTcRows + r] = l_run;
            mbar_arrive(lready);
            if constexpr (kPrefix) {
                if (__all_sync(0xffffffffu, mbar_wait(lready, vu & 1, err, abort_flag, p.wait_limit_ns))) {
                    tc::fence_after_sync();
                    // The plan kernel's partial slots and the partition pass's pieces.
                    griddep_wait();
                    const float l_pre = lsum[r] + lsum[kTcRows + r];
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + row_off) + hf * (D / 16);
                    if (!p.part_start) {
                        // One other piece per row, the suffix kernel's, in the row's own slot: the
                        // sequence's length, the piece's (max, sum) and this thread's half of its
                        // unnormalised output are loaded together, in one round trip.
                        const int len = p.context_lens[rseq];
                        const float2 ml = p.pml[row_id];
                        const float4* src = reinterpret_cast<const float4*>(p.pacc + row_id * D) + hf * (D / 8);
                        float4 pv[D / 8];
#pragma unroll
                        for (int e = 0; e < D / 8; ++e) pv[e] = src[e];
                        // A sequence the plan found invalid has no slot of its own: nothing is written.
                        const bool write = real && seq_len_valid(len, p.q_len, L, p.max_context_len, p.max_blocks_per_seq);
                        const float M = write ? fmaxf(m_run, ml.x) : m_run;
                        const float f0 = ex2(m_run - M);
                        float ltot = l_pre * f0;
                        const float fc = write ? ex2(ml.x - M) : 0.f;
                        if (write) ltot += ml.y * fc;
                        const float inv = 1.f / ltot;
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            uint32_t o[32];
                            tc::ld_x32(o_half + 32 * h, o);
                            float acc[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(o[e]) * f0;
                            if (write) {
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float4 v = pv[h * 8 + e];
                                    acc[4 * e] += v.x * fc;
                                    acc[4 * e + 1] += v.y * fc;
                                    acc[4 * e + 2] += v.z * fc;
                                    acc[4 * e + 3] += v.w * fc;
                                }
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    uint4 v;
                                    v.x = Elem<T>::pack(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
                                    v.y = Elem<T>::pack(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
                                    v.z = Elem<T>::pack(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
                                    v.w = Elem<T>::pack(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
                                    dst[h * 4 + c] = v;
                                }
                            }
                        }
                    } else {
                        // A sequence the plan found invalid has no slot of its own: nothing is written.
                        const bool write = real && seq_len_valid(p.context_lens[rseq], p.q_len, L, p.max_context_len,
                                                                 p.max_blocks_per_seq);
                        // The sequence's other pieces: partial slots part_start[i] + 1 .. (split-K
                        // partitions).
                        const long long slot0 = !write ? 0 : p.part_start[rseq];
                        // Merge the prefix piece (m_run, l_pre, O in TMEM) with the sequence's other
                        // pieces, in slot order, by their log-sum-exp, and write the output row.
                        const int npieces = !write ? 1 : p.part_start[rseq + 1] - (int)slot0;
                        const long long stride = (long long)p.q_len * p.num_heads;
                        const long long prow0 = (slot0 * p.q_len + t) * p.num_heads + hq;
                        float M = m_run;
                        for (int c = 1; c < npieces; ++c) M = fmaxf(M, p.pml[prow0 + c * stride].x);
                        const float f0 = ex2(m_run - M);
                        float ltot = l_pre * f0;
                        for (int c = 1; c < npieces; ++c) {
                            const float2 ml = p.pml[prow0 + c * stride];
                            ltot += ml.y * ex2(ml.x - M);
                        }
                        const float inv = 1.f / ltot;
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            uint32_t o[32];
                            tc::ld_x32(o_half + 32 * h, o);
                            float acc[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(o[e]) * f0;
                            for (int c = 1; c < npieces; ++c) {
                                const long long prow = prow0 + c * stride;
                                const float fc = ex2(p.pml[prow].x - M);
                                const float4* src = reinterpret_cast<const float4*>(p.pacc + prow * D) +
                                                    hf * (D / 8) + h * 8;
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const float4 v = src[e];
                                    acc[4 * e] += v.x * fc;
                                    acc[4 * e + 1] += v.y * fc;
                                    acc[4 * e + 2] += v.z * fc;
                                    acc[4 * e + 3] += v.w * fc;
                                }
                            }
                            if (write) {
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    uint4 v;
                                    v.x = Elem<T>::pack(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv);
                                    v.y = Elem<T>::pack(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv);
                                    v.z = Elem<T>::pack(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv);
                                    v.w = Elem<T>::pack(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv);
                                    dst[h * 4 + c] = v;
                                }
                            }
                        }
                    }
                }
            } else if (kMode == kModeSuffix && tile.blk0 > 0) {
                // A sequence with a shared prefix: its suffix piece (m, l, unnormalised O) goes to
                // partial slot i for the prefix kernel, which merges and writes the output.
                if (__all_sync(0xffffffffu, mbar_wait(lready, vu & 1, err, abort_flag, p.wait_limit_ns))) {
                    tc::fence_after_sync();
                    const long long prow = row_id;  // slot i: (i * q_len + t) * Hq + hq
                    if (real && hf == 0) p.pml_out[prow] = make_float2(m_run, lsum[r] + lsum[kTcRows + r]);
                    float4* dst = reinterpret_cast<float4*>(p.pacc_out + prow * D) + hf * (D / 8);
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        uint32_t o[32];
                        tc::ld_x32(o_half + 32 * h, o);
                        if (real) {
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                dst[h * 8 + c] =
                                    make_float4(__uint_as_float(o[4 * c]), __uint_as_float(o[4 * c + 1]),
                                                __uint_as_float(o[4 * c + 2]), __uint_as_float(o[4 * c + 3]));
                        }
                    }
                }
            } else if (__all_sync(0xffffffffu, mbar_wait(lready, vu & 1, err, abort_flag, p.wait_limit_ns))) {
                tc::fence_after_sync();
                const float inv = 1.f / (lsum[r] + lsum[kTcRows + r]);
                uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + row_off) + hf * (D / 16);
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    uint32_t o[32];
                    tc::ld_x32(o_half + 32 * h, o);
                    if (real) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 v;
                            v.x = Elem<T>::pack(__uint_as_float(o[8 * c + 0]) * inv, __uint_as_float(o[8 * c + 1]) * inv);
                            v.y = Elem<T>::pack(__uint_as_float(o[8 * c + 2]) * inv, __uint_as_float(o[8 * c + 3]) * inv);
                            v.z = Elem<T>::pack(__uint_as_float(o[8 * c + 4]) * inv, __uint_as_float(o[8 * c + 5]) * inv);
                            v.w = Elem<T>::pack(__uint_as_float(o[8 * c + 6]) * inv, __uint_as_float(o[8 * c + 7]) * inv);
                            dst[h * 4 + c] = v;
                        }
                    }
                }
            }
        }
        if (*abort_flag) ok = false;  // a wait of this unit gave up: no further unit
        gt_run += ntiles;
        ++vu_run;
        }
    }

    // Teardown: every TMEM access and product is complete; free TMEM.
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillTcParams p) {
    tc_attention<T, D, kModeChunk>(p, nullptr);
}

// The shared prefix of every prefix group once per kv head for all the group's query rows.
template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefix_tc_kernel(const __grid_constant__ PrefillTcParams p, const __grid_constant__ PrefixGroups g) {
    tc_attention<T, D, kModePrefix>(p, &g);
}

// Each sequence's chunk rows against its positions after its group's shared prefix (all of
// them for a sequence outside every group, which then gets its output here).
template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    suffix_tc_kernel(const __grid_constant__ PrefillTcParams p, const __grid_constant__ PrefixGroups g) {
    tc_attention<T, D, kModeSuffix>(p, &g);
}

// Suffix mode: the units ordered by their count of K/V tiles, longest first (a counting sort
// in one CTA; units of equal length in any order, which changes no result).  Bucket 0 holds
// the longest, 255 tiles or more, and invalid units count as empty.
constexpr int kOrderBuckets = 256;

__global__ void __launch_bounds__(1024) suffix_order_kernel(const __grid_constant__ PrefillTcParams p,
                                                            const __grid_constant__ PrefixGroups g) {
    __shared__ int start[kOrderBuckets];
    // Every earlier kernel first: the previous call's suffix kernel may still be reading the
    // order array, and the suffix kernel, which waits for this one, relies on the append.
    griddep_wait();
    griddep_launch_dependents();
    for (int b = threadIdx.x; b < kOrderBuckets; b += blockDim.x) start[b] = 0;
    __syncthreads();
    auto bucket = [&](int idx) {
        const TcTile t = tc_tile<kModeSuffix>(p, &g, idx);
        const int tiles = t.valid ? (t.nblk + kTcBlocks - 1) / kTcBlocks : 0;
        return kOrderBuckets - 1 - min(tiles, kOrderBuckets - 1);
    };
    for (int idx = threadIdx.x; idx < p.num_units; idx += blockDim.x) atomicAdd(&start[bucket(idx)], 1);
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive scan of the bucket counts: lane l holds buckets 8l .. 8l + 7
        constexpr int E = kOrderBuckets / 32;
        const int lane = threadIdx.x;
        int c[E], mine = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            c[e] = start[lane * E + e];
            mine += c[e];
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - mine;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            start[lane * E + e] = run;
            run += c[e];
        }
    }
    __syncthreads();
    int* order = const_cast<int*>(p.order);
    for (int idx = threadIdx.x; idx < p.num_units; idx += blockDim.x) order[atomicAdd(&start[bucket(idx)], 1)] = idx;
}

// Parameters shared by the chunk and prefix launches.
template <int D>
int tc_params(const DecodeArgs& a, PrefillTcParams& p) {
    if (int st = kv_tensor_map(&p.tmap_k, a.key_cache, a.dtype, a.num_blocks, a.num_kv_heads, D)) return st;
    if (int st = kv_tensor_map(&p.tmap_v, a.value_cache, a.dtype, a.num_blocks, a.num_kv_heads, D)) return st;
    p.out = a.out;
    p.query = a.query;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    if (int st = device_error_word(&p.err)) return st;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.num_blocks = (int)a.num_blocks;
    p.q_len = a.q_len;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.group = a.num_heads / a.num_kv_heads;
    p.total_rows = p.group * a.q_len;
    p.mtiles = (p.total_rows + kTcRows - 1) / kTcRows;
    p.max_context_len = a.max_context_len;
    const long long units = (long long)a.num_seqs * a.num_kv_heads * p.mtiles;
    if (units > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    p.num_units = (int)units;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.wait_limit_ns = static_cast<unsigned int>(wait_limit_ns());
    p.part_start = nullptr;
    p.pml = nullptr;
    p.pacc = nullptr;
    p.pml_out = nullptr;
    p.pacc_out = nullptr;
    p.order = nullptr;
    return PA_OK;
}

template <typename T, int D>
int launch_prefill_tc_typed(const DecodeArgs& a, cudaStream_t stream, int* launches) {
    PrefillTcParams p;
    if (int st = tc_params<D>(a, p)) return st;
    // One CTA per unit: the units of a prefill chunk are long and uneven (their causal ranges
    // differ by up to the chunk), and the hardware's hand-out of CTAs to SMs as they free up
    // balances them better than a fixed assignment of units to persistent CTAs (chunked-prefill
    // batch: 317 vs 359 us).
    const int grid = p.num_units;
    auto kfn = prefill_tc_kernel<T, D>;
    const int smem = TcLayout<D>::kAlloc;
    if (int st = ensure_dynamic_smem(reinterpret_cast<const void*>(kfn), smem)) return st;
    const int pc = profile_call_begin();
    profile_mark(pc, 0, stream);  // no plan kernel: marks 0 and 1 coincide
    profile_mark(pc, 1, stream);
    if (launch_pdl(kfn, dim3(grid), dim3(kTcThreads), (size_t)smem, stream, p) != cudaSuccess)
        return PA_ERR_CUDA;
    profile_mark(pc, 2, stream);
    profile_mark(pc, 3, stream);  // no merge kernel
    *launches += 1;
    return PA_OK;
}

template <typename T, int D>
int launch_prefix_tc_typed(const DecodeArgs& a, const int* part_start, const float2* pml, const float* pacc,
                           cudaStream_t stream, int* launches);

// A shared-prefix call entirely on tcgen05: the suffix kernel (one CTA per (sequence, kv head,
// 128-row tile) over the positions after the sequence's prefix; sequences outside every group
// get their output there), then the prefix kernel, which merges each grouped row's suffix piece
// (partial slot i) and writes the output.
template <typename T, int D>
int launch_shared_prefix_tc_typed(const DecodeArgs& a, float2* pml, float* pacc, int* order, cudaStream_t stream,
                                  int* launches) {
    PrefillTcParams p;
    if (int st = tc_params<D>(a, p)) return st;
    p.pml_out = pml;
    p.pacc_out = pacc;
    p.order = order;
    // Suffixes are a few tiles each: persistent CTAs (one per SM) save each unit the CTA's
    // set-up (barriers, tensor memory, first copies).
    int sms = 0;
    if (int st = sm_count(&sms)) return st;
    const int grid = PA_TC_SUFFIX_PERSISTENT ? std::min(p.num_units, sms) : p.num_units;
    auto sfn = suffix_tc_kernel<T, D>;
    const int smem = TcLayout<D>::kAlloc;
    if (int st = ensure_dynamic_smem(reinterpret_cast<const void*>(sfn), smem)) return st;
    const int pc = profile_call_begin();
    profile_mark(pc, 0, stream);
    // The persistent CTAs take the units longest first, back and forth across the CTAs.
    if (launch_pdl(suffix_order_kernel, dim3(1), dim3(1024), 0, stream, p, *a.groups) != cudaSuccess)
        return PA_ERR_CUDA;
    *launches += 1;
    profile_mark(pc, 1, stream);
    if (launch_pdl(sfn, dim3(grid), dim3(kTcThreads), (size_t)smem, stream, p, *a.groups) != cudaSuccess)
        return PA_ERR_CUDA;
    *launches += 1;
    profile_mark(pc, 2, stream);
    const int st = launch_prefix_tc_typed<T, D>(a, nullptr, pml, pacc, stream, launches);
    profile_mark(pc, 3, stream);
    return st;
}

template <typename T, int D>
int launch_prefix_tc_typed(const DecodeArgs& a, const int* part_start, const float2* pml, const float* pacc,
                           cudaStream_t stream, int* launches) {
    const PrefixGroups& g = *a.groups;
    if (g.tile_start[g.n] == 0) return PA_OK;
    PrefillTcParams p;
    if (int st = tc_params<D>(a, p)) return st;
    int sms = 0;
    if (int st = sm_count(&sms)) return st;
    const int grid = std::min(g.tile_start[g.n], sms);
    p.part_start = part_start;
    p.pml = pml;
    p.pacc = pacc;
    auto kfn = prefix_tc_kernel<T, D>;
    const int smem = TcLayout<D>::kAlloc;
    if (int st = ensure_dynamic_smem(reinterpret_cast<const void*>(kfn), smem)) return st;
    if (launch_pdl(kfn, dim3(grid), dim3(kTcThreads), (size_t)smem, stream, p, g) != cudaSuccess)
        return PA_ERR_CUDA;
    *launches += 1;
    return PA_OK;
}

}  // namespace

int launch_shared_prefix_tc(const DecodeArgs& a, float2* pml, float* pacc, int* order, cudaStream_t stream,
                            int* launches) {
    if (a.fp8 || !a.groups) return PA_ERR_UNSUPPORTED;
    if (a.dtype == PA_BF16) {
        if (a.head_dim == 128)
            return launch_shared_prefix_tc_typed<__nv_bfloat16, 128>(a, pml, pacc, order, stream, launches);
        if (a.head_dim == 64)
            return launch_shared_prefix_tc_typed<__nv_bfloat16, 64>(a, pml, pacc, order, stream, launches);
    } else {
        if (a.head_dim == 128) return launch_shared_prefix_tc_typed<__half, 128>(a, pml, pacc, order, stream, launches);
        if (a.head_dim == 64) return launch_shared_prefix_tc_typed<__half, 64>(a, pml, pacc, order, stream, launches);
    }
    return PA_ERR_UNSUPPORTED;
}

int launch_prefill_tc(const DecodeArgs& a, cudaStream_t stream, int* launches) {
    if (a.fp8) return PA_ERR_UNSUPPORTED;
    if (a.dtype == PA_BF16) {
        if (a.head_dim == 128) return launch_prefill_tc_typed<__nv_bfloat16, 128>(a, stream, launches);
        if (a.head_dim == 64) return launch_prefill_tc_typed<__nv_bfloat16, 64>(a, stream, launches);
    } else {
        if (a.head_dim == 128) return launch_prefill_tc_typed<__half, 128>(a, stream, launches);
        if (a.head_dim == 64) return launch_prefill_tc_typed<__half, 64>(a, stream, launches);
    }
    return PA_ERR_UNSUPPORTED;
}

int launch_prefix_tc(const DecodeArgs& a, const int* part_start, const float2* pml, const float* pacc,
                     cudaStream_t stream, int* launches) {
    if (a.fp8 || !a.groups) return PA_ERR_UNSUPPORTED;
    if (a.dtype == PA_BF16) {
        if (a.head_dim == 128)
            return launch_prefix_tc_typed<__nv_bfloat16, 128>(a, part_start, pml, pacc, stream, launches);
        if (a.head_dim == 64)
            return launch_prefix_tc_typed<__nv_bfloat16, 64>(a, part_start, pml, pacc, stream, launches);
    } else {
        if (a.head_dim == 128) return launch_prefix_tc_typed<__half, 128>(a, part_start, pml, pacc, stream, launches);
        if (a.head_dim == 64) return launch_prefix_tc_typed<__half, 64>(a, part_start, pml, pacc, stream, launches);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
