/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV decode attention
 * and the KV-append (reshape-and-cache) step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path; the two meet only in the
 * seeded input generator, which holds none of the arithmetic below.
 *
 * What it computes (sources are the three web pages the method is described
 * on; each page is cited by its title and section):
 *
 *  - Dense causal attention, "LLM 推理优化的系统视角", section 3.1 (KV Cache:
 *    what it reuses): O_t = softmax(Q_t K_{1:t}^T / sqrt(d_h)) V_{1:t}.
 *  - Blockwise (paged) attention equals that dense attention over the
 *    physical blocks concatenated in logical order: "每生成一个字都要把全部权重
 *    读一遍：从 vLLM 看 LLM 推理提速", section "KV Cache 又大又碎，为何不用操作
 *    系统分页的思路管它？", the equation s_j = q^T K_j / sqrt(d_k),
 *    o = sum_j softmax(s)_j V_j and the figure caption after it (physical
 *    placement does not change the result).  The oracle therefore first
 *    concatenates each sequence's blocks in logical order (walking its block
 *    table) and then runs the dense definition; there is no blocking, no
 *    online softmax and no split.
 *  - Block table: same page, same section (the per-request table mapping
 *    logical blocks to physical blocks, block size 16).
 *  - Query heads share K/V heads in contiguous groups (GQA): "LLM 推理优化的
 *    系统视角", section 3.2 (MHA / MQA / GQA list) and section 4.1.
 *  - Decode step reads the cached K/V and appends the new position's K/V:
 *    "LLM 推理优化的系统视角", section 3.1 (decode-step state change).  The
 *    append is a byte copy of row t into slot slot_mapping[t], the slot
 *    mapping being built in "prepare inputs" ("现代 LLM 推理引擎剖析", section
 *    1.6, Forward Pass 内部).
 *
 * Readings where the pages are silent:
 *  - context_lens[i] counts the tokens being decoded; the q_len query rows of
 *    sequence i are its last q_len positions, and row j attends positions
 *    0 .. L_i - q_len + j (causal inside the chunk).
 *  - kv head of query head h is h / (num_heads / num_kv_heads).
 *  - pool layout [num_blocks, block_size, num_kv_heads, head_dim], head_dim
 *    fastest; slot = physical_block * block_size + offset; slot < 0 = skip.
 *  - 16-bit storage: bf16 or IEEE fp16 bit patterns, widened exactly to fp64.
 *
 * PLANT: when compiled with -DPLANT=n (n > 0) one deliberate mistake is
 * planted, so that the test suite can show that its pins catch it.  The
 * product oracle is built with PLANT undefined.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef PLANT
#define PLANT 0
#endif

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

/* Exact widening of one 16-bit storage value to fp64. */
double oracle_bits_to_double(uint16_t bits, int dtype)
{
    if (dtype == ORACLE_BF16) {
        /* bf16 is the top half of an IEEE binary32 value. */
        uint32_t u = (uint32_t)bits << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int frac = bits & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);                 /* zero / subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    }
    return sign ? -v : v;
}

/* Vector form, used by the tests to pin the widening against library casts. */
void oracle_bits_to_double_vec(const uint16_t* bits, int64_t n, int dtype, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bits_to_double(bits[i], dtype);
}

/*
 * Gather sequence i's K (or V) in logical order: token p lives in physical
 * block block_table[p / block_size] at offset p % block_size.
 * dst: [L, num_kv_heads, head_dim] fp64.  Returns 0, or -1 if a block id used
 * by the sequence is outside [0, num_blocks).
 */
static int gather_sequence(const uint16_t* cache, const int32_t* table, int L,
                           int num_kv_heads, int head_dim, int block_size,
                           int64_t num_blocks, int dtype, double* dst)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int p = 0; p < L; ++p) {
        int32_t blk = table[p / block_size];
        int off = p % block_size;
#if PLANT == 4
        off = block_size - 1 - off;                   /* planted: offset reversed in block */
#endif
        if (blk < 0 || (int64_t)blk >= num_blocks) return -1;
        const uint16_t* src = cache + ((int64_t)blk * block_size + off) * row;
        for (int64_t e = 0; e < row; ++e) dst[(int64_t)p * row + e] = oracle_bits_to_double(src[e], dtype);
    }
    return 0;
}

/*
 * Paged decode attention, fp64.
 *   out          [num_seqs, q_len, num_heads, head_dim] fp64 (written)
 *   query        [num_seqs, q_len, num_heads, head_dim] 16-bit
 *   key_cache    [num_blocks, block_size, num_kv_heads, head_dim] 16-bit
 *   value_cache  same as key_cache
 *   block_tables [num_seqs, max_blocks_per_seq] int32
 *   context_lens [num_seqs] int32 (includes the q_len positions being decoded)
 * Sequences whose length is < q_len, or whose block table points outside the
 * pool, get NaN outputs; the return value counts them.
 * num_threads <= 0 uses the OpenMP default.
 */
int oracle_decode_attention(double* out, const uint16_t* query,
                            const uint16_t* key_cache, const uint16_t* value_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int q_len,
                            int num_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, double scale,
                            int dtype, int num_threads)
{
    const int group = num_heads / num_kv_heads;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int i = 0; i < num_seqs; ++i) {
        const int L = context_lens[i];
        double* o_seq = out + (int64_t)i * q_len * num_heads * head_dim;
        int ok = (L >= q_len && L >= 1 && head_dim <= 1024 &&
                  (L + block_size - 1) / block_size <= max_blocks_per_seq);
        double *K = NULL, *V = NULL, *s = NULL;
        if (ok) {
            const int64_t n = (int64_t)L * num_kv_heads * head_dim;
            K = (double*)malloc(sizeof(double) * n);
            V = (double*)malloc(sizeof(double) * n);
            s = (double*)malloc(sizeof(double) * L);
            const int32_t* table = block_tables + (int64_t)i * max_blocks_per_seq;
            /* Step 1: concatenate the physical blocks in logical order. */
            ok = K && V && s &&
                 gather_sequence(key_cache, table, L, num_kv_heads, head_dim, block_size, num_blocks, dtype, K) == 0 &&
                 gather_sequence(value_cache, table, L, num_kv_heads, head_dim, block_size, num_blocks, dtype, V) == 0;
#if PLANT == 7
            if (ok) memcpy(V, K, sizeof(double) * n);      /* planted: V read from the K cache */
#endif
        }
        if (!ok) {
            for (int64_t e = 0; e < (int64_t)q_len * num_heads * head_dim; ++e) o_seq[e] = NAN;
            bad += 1;
            free(K); free(V); free(s);
            continue;
        }
        /* Step 2: dense causal attention for every query row and head. */
        for (int j = 0; j < q_len; ++j) {
            int last = L - q_len + j;                         /* last position row j may attend */
#if PLANT == 3
            last = last - 1 < 0 ? 0 : last - 1;               /* planted: causal limit off by one */
#elif PLANT == 6
            last = L - 1 - j;                                 /* planted: chunk rows reversed */
#endif
            for (int h = 0; h < num_heads; ++h) {
                int kvh = h / group;
#if PLANT == 2
                kvh = h % num_kv_heads;                       /* planted: interleaved head groups */
#endif
                const uint16_t* qrow = query + (((int64_t)i * q_len + j) * num_heads + h) * head_dim;
                double* o = o_seq + ((int64_t)j * num_heads + h) * head_dim;
                double qd[1024];
                double sc = scale;
#if PLANT == 1
                sc = 1.0;                                     /* planted: scale dropped */
#endif
                for (int k = 0; k < head_dim; ++k) qd[k] = oracle_bits_to_double(qrow[k], dtype);
                /* scores s_p = scale * q . K_p for p = 0 .. last */
                double m = -INFINITY;
                for (int p = 0; p <= last; ++p) {
                    const double* kp = K + ((int64_t)p * num_kv_heads + kvh) * head_dim;
                    double dot = 0.0;
                    for (int k = 0; k < head_dim; ++k) dot += qd[k] * kp[k];
                    s[p] = sc * dot;
                    if (s[p] > m) m = s[p];
                }
                /* softmax weights and the weighted sum of V rows */
                double den = 0.0;
                for (int p = 0; p <= last; ++p) {
                    s[p] = exp(s[p] - m);
#if PLANT == 5
                    if (p == last && last > 0) continue;      /* planted: last weight left out of the sum */
#endif
                    den += s[p];
                }
                for (int k = 0; k < head_dim; ++k) o[k] = 0.0;
                for (int p = 0; p <= last; ++p) {
                    const double* vp = V + ((int64_t)p * num_kv_heads + kvh) * head_dim;
                    for (int k = 0; k < head_dim; ++k) o[k] += s[p] * vp[k];
                }
                for (int k = 0; k < head_dim; ++k) o[k] /= den;
            }
        }
        free(K); free(V); free(s);
    }
    return bad;
}

/*
 * KV append: for each new token t with slot_mapping[t] >= 0, copy its
 * [num_kv_heads, head_dim] K row and V row byte for byte into
 * cache[slot / block_size, slot % block_size].  Returns the number of tokens
 * whose slot lies beyond the pool (those are not written).
 */
int oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                             uint16_t* key_cache, uint16_t* value_cache,
                             const int64_t* slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                              /* padding token: nothing to write */
        if (slot >= num_blocks * block_size) { ++bad; continue; }
#if PLANT == 14
        int64_t blk = slot % block_size, off = slot / block_size;   /* planted: block and offset swapped */
        if (blk >= num_blocks || off >= block_size) { ++bad; continue; }
#else
        int64_t blk = slot / block_size, off = slot % block_size;
#endif
        uint16_t* kd = key_cache + (blk * block_size + off) * row;
        uint16_t* vd = value_cache + (blk * block_size + off) * row;
        memcpy(kd, key + t * row, sizeof(uint16_t) * row);
        memcpy(vd, value + t * row, sizeof(uint16_t) * row);
    }
    return bad;
}

/*
 * Copy-on-write block copy ("每生成一个字都要把全部权重读一遍：从 vLLM 看 LLM 推理提速",
 * paged-KV section, the reference-count paragraph: a sequence about to write into a
 * block it shares first gets its own copy of that block).  For every pair
 * (src, dst) of block_mapping [num_pairs, 2], the whole K block and V block
 * [block_size, num_kv_heads, head_dim] are copied byte for byte from src to dst.
 * Pairs with an id outside [0, num_blocks) are skipped and counted in the return
 * value.  Pairs are applied in order.
 */
int oracle_copy_blocks(uint16_t* key_cache, uint16_t* value_cache, const int64_t* block_mapping,
                       int64_t num_pairs, int num_kv_heads, int head_dim, int block_size,
                       int64_t num_blocks)
{
    const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
    int bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = block_mapping[2 * i], dst = block_mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++bad; continue; }
#if PLANT == 12
        int64_t tmp = src; src = dst; dst = tmp;                   /* planted: copied the wrong way */
#endif
        memmove(key_cache + dst * blk, key_cache + src * blk, sizeof(uint16_t) * blk);
        memmove(value_cache + dst * blk, value_cache + src * blk, sizeof(uint16_t) * blk);
    }
    return bad;
}

/*
 * Speculative-decoding verification ("现代 LLM 推理引擎剖析", section 2.4 Speculative
 * Decoding, steps 3 and 4; the gamma + 1 positions of "每生成一个字都要把全部权重读一遍",
 * section "对症下药").  For each sequence, with k draft tokens:
 *   scan i = 0 .. k-1 left to right, t = draft_tokens[i]:
 *     accept if p_large[i][t] >= p_draft[i][t];
 *     else accept if u_accept[i] < p_large[i][t] / p_draft[i][t]  (probability p_large/p_draft);
 *     at the first rejection stop and draw one token from (p_large[i] - p_draft[i])+;
 *   if all k are accepted, draw a bonus token from p_large[k].
 * A draw from weights w[0..V) with uniform u takes the smallest v whose prefix sum
 * of w exceeds u times the total.  Reading (the pages give no sampling procedure):
 * the weights are fp32; each is converted exactly to a fixed-point integer
 * floor(w * 2^40), u to floor(u * 2^24), the threshold is floor(u24 * total / 2^24),
 * so prefix sums are integer-exact and independent of summation order.  A residual
 * whose integer total is 0 falls back to p_large[i].
 * Outputs: num_accepted[n] in [0, k]; out_tokens[n][0..k]: the accepted drafts,
 * then the drawn token, then -1.
 */
static uint64_t fixed40(float w) { return (uint64_t)floor((double)w * 1099511627776.0); }  /* 2^40 */

static int draw_fixed(const float* a, const float* b, int vocab, float u)
{
    /* weights a - b clamped at 0 (b == NULL: a itself) */
    uint64_t total = 0;
    for (int v = 0; v < vocab; ++v) {
#if PLANT == 9
        float w = b ? b[v] - a[v] : a[v];   /* planted: residual taken the wrong way round */
#else
        float w = b ? a[v] - b[v] : a[v];
#endif
        if (!(w > 0.0f)) w = 0.0f;
        total += fixed40(w);
    }
    if (total == 0) return -1;
    uint64_t u24 = (uint64_t)floor((double)u * 16777216.0);          /* 2^24 */
    unsigned __int128 prod = (unsigned __int128)u24 * total;
    uint64_t thresh = (uint64_t)(prod >> 24);
    uint64_t run = 0;
    for (int v = 0; v < vocab; ++v) {
        float w = b ? a[v] - b[v] : a[v];
        if (!(w > 0.0f)) w = 0.0f;
#if PLANT == 9
        w = b ? b[v] - a[v] : a[v];
        if (!(w > 0.0f)) w = 0.0f;
#endif
        run += fixed40(w);
        if (run > thresh) return v;
    }
    return vocab - 1;
}

int oracle_spec_verify(int32_t* num_accepted, int32_t* out_tokens, const float* target_probs,
                       const float* draft_probs, const int32_t* draft_tokens, const float* u_accept,
                       const float* u_sample, int num_seqs, int k, int vocab)
{
    for (int n = 0; n < num_seqs; ++n) {
        const float* pl = target_probs + (int64_t)n * (k + 1) * vocab;
        const float* pd = draft_probs + (int64_t)n * k * vocab;
        int32_t* out = out_tokens + (int64_t)n * (k + 1);
        int i = 0;
        for (; i < k; ++i) {
            int t = draft_tokens[(int64_t)n * k + i];
            float a = pl[(int64_t)i * vocab + t], b = pd[(int64_t)i * vocab + t];
            int accept = a >= b;
            if (!accept) {
#if PLANT == 8
                volatile float ratio = b / a;   /* planted: ratio inverted */
#else
                volatile float ratio = a / b;   /* IEEE single-precision division */
#endif
                accept = u_accept[(int64_t)n * k + i] < ratio;
            }
            if (!accept) break;
            out[i] = t;
        }
        int tok;
        if (i < k) {
            tok = draw_fixed(pl + (int64_t)i * vocab, pd + (int64_t)i * vocab, vocab, u_sample[n]);
            if (tok < 0) tok = draw_fixed(pl + (int64_t)i * vocab, NULL, vocab, u_sample[n]);
        } else {
            tok = draw_fixed(pl + (int64_t)k * vocab, NULL, vocab, u_sample[n]);
        }
        out[i] = tok;
        for (int j = i + 1; j <= k; ++j) out[j] = -1;
        num_accepted[n] = i;
    }
    return 0;
}

/*
 * FP8 KV cache ("LLM 推理优化的系统视角", section 4.1: quantising the KV cache reduces its
 * bytes).  Reading (the pages fix no format): OCP FP8 E4M3 (1 sign, 4 exponent bits,
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448) with
 * one fp32 scale per cache tensor; stored byte = e4m3(x / scale) with the quotient in
 * fp32 and rounded to nearest even, saturating to +-448; read value = e4m3 * scale.
 */
static double round_half_even(double x)
{
    double f = floor(x), d = x - f;
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

uint8_t oracle_e4m3_encode(float v)
{
    if (v != v) return 0x7f;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    const double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7e;                       /* saturate */
    if (a < ldexp(1.0, -6)) {                                 /* subnormal: units of 2^-9 */
        double r = round_half_even(a / ldexp(1.0, -9));
        return sign | (uint8_t)r;                             /* r == 8 is exponent field 1, mantissa 0 */
    }
    int E;
    frexp(a, &E);                                             /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;                                            /* a in [2^e, 2^(e+1)) */
#if PLANT == 11
    double r = floor((a / ldexp(1.0, e) - 1.0) * 8.0);         /* planted: truncation, not round-to-even */
#else
    double r = round_half_even((a / ldexp(1.0, e) - 1.0) * 8.0);
#endif
    if (r == 8.0) { e += 1; r = 0.0; }
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)r;
}

double oracle_e4m3_decode(uint8_t b)
{
    const int sign = b >> 7, field = (b >> 3) & 0xf, mant = b & 7;
    double v;
    if (field == 15 && mant == 7) return NAN;
    if (field == 0) v = ldexp((double)mant, -9);
#if PLANT == 10
    else v = ldexp(1.0 + mant / 8.0, field - 8);               /* planted: exponent bias 8 */
#else
    else v = ldexp(1.0 + mant / 8.0, field - 7);
#endif
    return sign ? -v : v;
}

void oracle_e4m3_encode_vec(const float* x, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_vec(const uint8_t* b, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(b[i]);
}

/* Append into FP8 caches: row t of key / value (16-bit, dtype) quantised with the scales. */
int oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, uint8_t* key_cache,
                                 uint8_t* value_cache, const int64_t* slot_mapping, int64_t num_tokens,
                                 int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                                 int dtype, float k_scale, float v_scale)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) { ++bad; continue; }
        for (int64_t e = 0; e < row; ++e) {
            float k = (float)oracle_bits_to_double(key[t * row + e], dtype);
            float v = (float)oracle_bits_to_double(value[t * row + e], dtype);
            key_cache[slot * row + e] = oracle_e4m3_encode(k / k_scale);
            value_cache[slot * row + e] = oracle_e4m3_encode(v / v_scale);
        }
    }
    return bad;
}

/*
 * Paged decode attention over FP8 caches: as oracle_decode_attention, with every K
 * element read as e4m3 * k_scale and every V element as e4m3 * v_scale (fp64).
 */
int oracle_decode_attention_fp8(double* out, const uint16_t* query, const uint8_t* key_cache,
                                const uint8_t* value_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                                int q_len, int num_heads, int num_kv_heads, int head_dim,
                                int block_size, int64_t num_blocks, double scale, int dtype,
                                float k_scale, float v_scale, int num_threads)
{
    const int group = num_heads / num_kv_heads;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    int bad = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int i = 0; i < num_seqs; ++i) {
        const int L = context_lens[i];
        double* o_seq = out + (int64_t)i * q_len * num_heads * head_dim;
        int ok = L >= q_len && L >= 1 && head_dim <= 1024 && (L + block_size - 1) / block_size <= max_blocks_per_seq;
        double *K = NULL, *V = NULL, *s = NULL;
        if (ok) {
            K = (double*)malloc(sizeof(double) * L * row);
            V = (double*)malloc(sizeof(double) * L * row);
            s = (double*)malloc(sizeof(double) * L);
            const int32_t* table = block_tables + (int64_t)i * max_blocks_per_seq;
            ok = K && V && s;
            /* concatenate the blocks in logical order, dequantising */
            for (int p = 0; ok && p < L; ++p) {
                int32_t blk = table[p / block_size];
                if (blk < 0 || (int64_t)blk >= num_blocks) { ok = 0; break; }
                const int64_t base = ((int64_t)blk * block_size + p % block_size) * row;
                for (int64_t e = 0; e < row; ++e) {
#if PLANT == 13
                    K[(int64_t)p * row + e] = oracle_e4m3_decode(key_cache[base + e]) * (double)v_scale;  /* planted */
                    V[(int64_t)p * row + e] = oracle_e4m3_decode(value_cache[base + e]) * (double)k_scale;
#else
                    K[(int64_t)p * row + e] = oracle_e4m3_decode(key_cache[base + e]) * (double)k_scale;
                    V[(int64_t)p * row + e] = oracle_e4m3_decode(value_cache[base + e]) * (double)v_scale;
#endif
                }
            }
        }
        if (!ok) {
            for (int64_t e = 0; e < (int64_t)q_len * num_heads * head_dim; ++e) o_seq[e] = NAN;
            bad += 1;
            free(K); free(V); free(s);
            continue;
        }
        for (int j = 0; j < q_len; ++j) {
            const int last = L - q_len + j;
            for (int h = 0; h < num_heads; ++h) {
                const int kvh = h / group;
                const uint16_t* qrow = query + (((int64_t)i * q_len + j) * num_heads + h) * head_dim;
                double* o = o_seq + ((int64_t)j * num_heads + h) * head_dim;
                double qd[1024];
                for (int k = 0; k < head_dim; ++k) qd[k] = oracle_bits_to_double(qrow[k], dtype);
                double m = -INFINITY;
                for (int p = 0; p <= last; ++p) {
                    const double* kp = K + ((int64_t)p * num_kv_heads + kvh) * head_dim;
                    double dot = 0.0;
                    for (int k = 0; k < head_dim; ++k) dot += qd[k] * kp[k];
                    s[p] = scale * dot;
                    if (s[p] > m) m = s[p];
                }
                double den = 0.0;
                for (int p = 0; p <= last; ++p) { s[p] = exp(s[p] - m); den += s[p]; }
                for (int k = 0; k < head_dim; ++k) o[k] = 0.0;
                for (int p = 0; p <= last; ++p) {
                    const double* vp = V + ((int64_t)p * num_kv_heads + kvh) * head_dim;
                    for (int k = 0; k < head_dim; ++k) o[k] += s[p] * vp[k];
                }
                for (int k = 0; k < head_dim; ++k) o[k] /= den;
            }
        }
        free(K); free(V); free(s);
    }
    return bad;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
