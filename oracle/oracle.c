/*
 * oracle.c -- plain, slow, obviously-correct CPU statement of the DeepSeek-V3.2
 * sparse-attention indexer hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library; the two meet only on the seeded inputs.
 *
 * Every function states the definition it follows.  Sources (web pages):
 *   [GATHER]  vLLM PR #25869 "[Model] Support Deepseek V3.2", code review of
 *             cp_gather_indexer_k_quant_cache (per-request loop: full blocks,
 *             then the partial last block; indexer-K block = block_size x
 *             head_dim fp8 values followed by block_size fp32 scales).
 *   [FALLBK]  vLLM PR #36250 "[kernel] Fix FP8 paged MQA fallback for CUDA
 *             graph capture": the paged MQA logits op over context_lens and
 *             the optional -inf tail (clean_logits, review thread).
 *   [DSMLA]   vLLM PR #47090 (prhub summary), "key source snippet" of
 *             _fused_norm_rope_kernel, fp8_ds_mla branch: 656 B entry
 *             [512 B fp8 NoPE][4 x fp32 tile scales][64 x bf16 RoPE],
 *             tile_scale = max(amax * (1/448), 1.1754944e-38), fp8 = x / scale.
 *   [ATOM]    ROCm/ATOM PR #1094 "[Feat] Support DSv3.2 with sglang-ATOM plugin
 *             and sglang sparse MLA", Technical Details: per-query top-k into a
 *             2-D index buffer, request-local top-k indices converted to global
 *             paged-KV indices.
 *   [SCORE]   The DeepSeek-V3.2 lightning-indexer score:
 *             logit[t,s] = k_scale[s] * sum_h w[t,h] * ReLU(q[t,h,:] . k[s,:]);
 *             indexer K quantised per token, scale = amax / 448.
 *   [OCP]     OCP 8-bit floating point specification, E4M3: bias 7, no
 *             infinities, S.1111.111 is NaN, largest finite 448.
 *   [DSMLA] also names the step this branch belongs to: the fused RMSNorm +
 *             RoPE + cache write of one token (the norm and rotation formulas are
 *             not printed there; the readings sit with the function).
 *
 * Readings of points the pages leave open (each also listed in the design notes):
 *   - fp8 rounding is round-to-nearest-even, saturating to +-448.
 *   - indexer K: scale = amax / 448 (IEEE f32 division), floored at FLT_MIN so
 *     that an all-zero token yields zero codes; codes = enc(x / scale) with an
 *     IEEE f32 division.
 *   - a negative slot_mapping entry means "skip this token".
 *   - decode row (b, j) of next_n sees L = context_lens[b] - next_n + 1 + j keys.
 *   - logits are computed exactly (every e4m3 product is a multiple of 2^-18 and
 *     |q.k| < 2^25, so a double sum is exact and order-free), weighted in double,
 *     then rounded once to f32.
 *   - top-k: order by (value desc, index asc), -0.0 equals +0.0, take
 *     min(k, L), emit in ascending index order, pad with -1; remap
 *     g = block_table[b, s / bs] * bs + s % bs, -1 stays -1.
 *   - sparse MLA decode: softmax attention of the bf16 query over the
 *     dequantised entries its global indices name (the reading sits with the
 *     function).
 *
 * Build: gcc -O3 -fopenmp -fPIC -shared (no -ffast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* OCP FP8 E4M3 codec [OCP]                                                   */
/* ------------------------------------------------------------------------- */

/* Exact value of an E4M3 code.  Normal: 2^(e-7) * (1 + m/8), e in 1..15;
 * subnormal: 2^-6 * (m/8); S.1111.111 is NaN. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Non-negative finite codes 0x00..0x7E in increasing value order (the code
 * order is the value order for a fixed sign). */
static double g_pos_values[127];
static int g_codec_ready = 0;

static void codec_init(void)
{
    if (g_codec_ready) return;
    for (int c = 0; c < 127; ++c) g_pos_values[c] = oracle_e4m3_decode((uint8_t)c);
    g_codec_ready = 1;
}

/* Round-to-nearest, ties to the even code (mantissa LSB 0); magnitudes at or
 * beyond 448 saturate to 448; NaN maps to the NaN code. */
uint8_t oracle_e4m3_encode(float x)
{
    codec_init();
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* largest code lo with value <= a (value(0) = 0 <= a always) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_pos_values[mid] <= a) lo = mid; else hi = mid - 1;
    }
    int c;
    if (g_pos_values[lo] == a) {
        c = lo;
    } else {
        /* lo < 126 here because a < 448 = value(126) */
        double below = a - g_pos_values[lo];      /* exact: see header */
        double above = g_pos_values[lo + 1] - a;  /* exact */
        if (below < above) c = lo;
        else if (above < below) c = lo + 1;
        else c = (lo % 2 == 0) ? lo : lo + 1;
    }
    return (uint8_t)(sign | c);
}

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------- */
/* Indexer K quantise + paged cache write [GATHER layout] [SCORE scale]       */
/* ------------------------------------------------------------------------- */

/* cache: uint8 [num_blocks, block_size * (head_dim + 4)].  Token at slot
 * (blk, off): fp8 values at blk*B + off*head_dim, fp32 scale at
 * blk*B + block_size*head_dim + 4*off.  Returns 0, or -1 on a slot past the
 * pool. */
int oracle_quant_write_k(const uint16_t* k_bf16, int64_t n, int head_dim,
                         const int64_t* slot_mapping, uint8_t* cache,
                         int64_t num_blocks, int block_size)
{
    codec_init();
    const int64_t block_bytes = (int64_t)block_size * (head_dim + 4);
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < n; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        if (blk >= num_blocks) { bad = 1; continue; }
        const uint16_t* src = k_bf16 + t * head_dim;
        float amax = 0.0f;
        for (int i = 0; i < head_dim; ++i) {
            float a = fabsf(bf16_to_f32(src[i]));
            if (a > amax) amax = a;
        }
        float scale = amax / 448.0f;
        if (!(scale >= FLT_MIN)) scale = FLT_MIN;
        uint8_t* base = cache + blk * block_bytes;
        for (int i = 0; i < head_dim; ++i) {
            float x = bf16_to_f32(src[i]);
            float y = x / scale;
            base[off * head_dim + i] = oracle_e4m3_encode(y);
        }
        memcpy(base + (int64_t)block_size * head_dim + 4 * off, &scale, 4);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Paged gather into contiguous K [GATHER]                                    */
/* ------------------------------------------------------------------------- */

/* For each request b with s = cu[b+1]-cu[b] > 0: copy its full blocks, then
 * the first `remaining` rows of its last block, into out_k[cu[b]:] (fp8 rows of
 * head_dim bytes) and out_scale[cu[b]:] (fp32).  Empty requests are skipped;
 * rows past cu[batch] are not touched. */
int oracle_gather_k(const uint8_t* cache, int64_t num_blocks, int block_size,
                    int head_dim, const int32_t* block_table, int64_t bt_stride,
                    const int32_t* cu_seq_lens, int batch, uint8_t* out_k,
                    float* out_scale)
{
    const int64_t block_bytes = (int64_t)block_size * (head_dim + 4);
    const int64_t val_bytes = (int64_t)block_size * head_dim;
    for (int b = 0; b < batch; ++b) {
        int64_t s = (int64_t)cu_seq_lens[b + 1] - cu_seq_lens[b];
        if (s <= 0) continue;
        int64_t start = cu_seq_lens[b];
        int64_t tot = (s + block_size - 1) / block_size;
        const int32_t* blocks = block_table + (int64_t)b * bt_stride;
        int64_t num_full = s / block_size;
        for (int64_t i = 0; i < num_full; ++i) {
            int64_t blk = blocks[i];
            if (blk < 0 || blk >= num_blocks) return -1;
            const uint8_t* src = cache + blk * block_bytes;
            memcpy(out_k + (start + i * block_size) * head_dim, src, (size_t)val_bytes);
            memcpy(out_scale + start + i * block_size, src + val_bytes, (size_t)block_size * 4);
        }
        int64_t remaining = s - num_full * block_size;
        if (remaining > 0) {
            int64_t blk = blocks[tot - 1];
            if (blk < 0 || blk >= num_blocks) return -1;
            const uint8_t* src = cache + blk * block_bytes;
            int64_t dst = start + num_full * block_size;
            memcpy(out_k + dst * head_dim, src, (size_t)(remaining * head_dim));
            memcpy(out_scale + dst, src + val_bytes, (size_t)(remaining * 4));
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* MQA logits [SCORE] [FALLBK]                                                */
/* ------------------------------------------------------------------------- */

/* One score: k_scale * sum_h w_h * max(q_h . k, 0); the dot products are
 * exact in double, the head sum is taken in double in head order. */
static float score_one(const double* qd /*[heads*head_dim]*/, const float* w,
                       const double* kd /*[head_dim]*/, float kscale, int heads,
                       int head_dim)
{
    double acc = 0.0;
    for (int h = 0; h < heads; ++h) {
        const double* qh = qd + (int64_t)h * head_dim;
        double d = 0.0;
        for (int i = 0; i < head_dim; ++i) d += qh[i] * kd[i];
        if (d > 0.0) acc += (double)w[h] * d;
    }
    return (float)((double)kscale * acc);
}

static void decode_row(const uint8_t* src, double* dst, int64_t n, const double* table)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = table[src[i]];
}

static void build_table(double* table)
{
    for (int c = 0; c < 256; ++c) table[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Decode (paged) logits.  Row r = b*next_n + j sees
 * L = context_lens[b] - next_n + 1 + j keys (clamped to [0, ld]); key s lives
 * in block block_table[b, s/bs] at offset s%bs.  logits is [nrows_out, ld];
 * out row i is logical row rows[i] (or i when rows is NULL).  Entries in
 * [L, ld) are -inf when clean is non-zero, else untouched. */
int oracle_paged_mqa_logits(const uint8_t* q, const float* w, const uint8_t* cache,
                            int64_t num_blocks, int block_size,
                            const int32_t* context_lens, const int32_t* block_table,
                            int64_t bt_stride, int batch, int next_n, int heads,
                            int head_dim, float* logits, int64_t ld, int clean,
                            const int64_t* rows, int64_t nrows)
{
    double table[256];
    build_table(table);
    const int64_t block_bytes = (int64_t)block_size * (head_dim + 4);
    const int64_t total_rows = (int64_t)batch * next_n;
    const int64_t nout = rows ? nrows : total_rows;
    const int64_t qrow = (int64_t)heads * head_dim;
    int bad = 0;
    if (head_dim > 512) return -2;
    double* qd = (double*)malloc(sizeof(double) * qrow);
    if (!qd) return -2;
    for (int64_t i = 0; i < nout; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= total_rows) { bad = 1; continue; }
        int64_t b = r / next_n, j = r % next_n;
        int64_t L = (int64_t)context_lens[b] - next_n + 1 + j;
        if (L < 0) L = 0;
        if (L > ld) { bad = 1; L = ld; }
        decode_row(q + r * qrow, qd, qrow, table);
        const float* wr = w + r * heads;
        float* out = logits + i * ld;
#pragma omp parallel for schedule(static) reduction(| : bad)
        for (int64_t s = 0; s < L; ++s) {
            int64_t blk = block_table[b * bt_stride + s / block_size];
            if (blk < 0 || blk >= num_blocks) { bad = 1; continue; }
            int64_t off = s % block_size;
            const uint8_t* base = cache + blk * block_bytes;
            double kd[512];
            decode_row(base + off * head_dim, kd, head_dim, table);
            float ks;
            memcpy(&ks, base + (int64_t)block_size * head_dim + 4 * off, 4);
            out[s] = score_one(qd, wr, kd, ks, heads, head_dim);
        }
        if (clean)
            for (int64_t s = L; s < ld; ++s) out[s] = -INFINITY;
    }
    free(qd);
    return bad ? -1 : 0;
}

/* Prefill (contiguous K) logits.  Row t sees keys [ks[t], ke[t]); column j of
 * the row is key ks[t] + j.  Same output convention as above. */
int oracle_mqa_logits(const uint8_t* q, const float* w, const uint8_t* k,
                      const float* k_scale, const int32_t* ks, const int32_t* ke,
                      int64_t tq, int64_t tk, int heads, int head_dim, float* logits,
                      int64_t ld, int clean, const int64_t* rows, int64_t nrows)
{
    double table[256];
    build_table(table);
    const int64_t nout = rows ? nrows : tq;
    const int64_t qrow = (int64_t)heads * head_dim;
    int bad = 0;
    if (head_dim > 512) return -2;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < nout; ++i) {
        int64_t t = rows ? rows[i] : i;
        if (t < 0 || t >= tq) { bad = 1; continue; }
        int64_t s0 = ks[t], s1 = ke[t];
        if (s0 < 0 || s1 > tk) { bad = 1; continue; }
        int64_t n = s1 - s0;
        if (n < 0) n = 0;
        if (n > ld) { bad = 1; n = ld; }
        double* qd = (double*)malloc(sizeof(double) * qrow);
        double kd[512];
        if (!qd) { bad = 1; continue; }
        decode_row(q + t * qrow, qd, qrow, table);
        float* out = logits + i * ld;
        for (int64_t j = 0; j < n; ++j) {
            decode_row(k + (s0 + j) * head_dim, kd, head_dim, table);
            out[j] = score_one(qd, w + t * heads, kd, k_scale[s0 + j], heads, head_dim);
        }
        if (clean)
            for (int64_t j = n; j < ld; ++j) out[j] = -INFINITY;
        free(qd);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Top-k selection + global remap [ATOM]                                      */
/* ------------------------------------------------------------------------- */

typedef struct { float v; int32_t i; } vi_t;

/* (value descending, index ascending); C float compare treats -0.0 == +0.0 */
static int cmp_value_desc(const void* pa, const void* pb)
{
    const vi_t* a = (const vi_t*)pa;
    const vi_t* b = (const vi_t*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int cmp_int_asc(const void* pa, const void* pb)
{
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* Row r (length L = row_len[r], request row_req[r]): pick the min(k, L)
 * columns with the largest logits (ties to the lower index), write them in
 * ascending index order, pad with -1, and map each to its global paged slot. */
int oracle_topk_to_global(const float* logits, int64_t ld, int64_t rows,
                          const int32_t* row_len, const int32_t* row_req,
                          const int32_t* block_table, int64_t bt_stride,
                          int block_size, int k, int32_t* out_local,
                          int32_t* out_global)
{
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t L = row_len[r];
        if (L < 0) L = 0;
        if (L > ld) { bad = 1; L = ld; }
        vi_t* buf = (vi_t*)malloc(sizeof(vi_t) * (L > 0 ? L : 1));
        int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (k > 0 ? k : 1));
        if (!buf || !sel) { bad = 1; free(buf); free(sel); continue; }
        for (int64_t s = 0; s < L; ++s) { buf[s].v = logits[r * ld + s]; buf[s].i = (int32_t)s; }
        qsort(buf, (size_t)L, sizeof(vi_t), cmp_value_desc);
        int64_t m = L < k ? L : k;
        for (int64_t i = 0; i < m; ++i) sel[i] = buf[i].i;
        qsort(sel, (size_t)m, sizeof(int32_t), cmp_int_asc);
        int64_t b = row_req[r];
        for (int64_t i = 0; i < k; ++i) {
            int32_t s = i < m ? sel[i] : -1;
            int32_t g = -1;
            if (s >= 0) {
                int64_t blk = block_table[b * bt_stride + s / block_size];
                g = (int32_t)(blk * block_size + s % block_size);
            }
            if (out_local) out_local[r * k + i] = s;
            out_global[r * k + i] = g;
        }
        free(buf);
        free(sel);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* fp8_ds_mla cache write [DSMLA]                                             */
/* ------------------------------------------------------------------------- */

/* Entry at blk*block_stride + off*entry_stride (bytes):
 *   [0,512)   fp8 NoPE, 4 tiles of 128, each coded with its own scale
 *   [512,528) the 4 fp32 tile scales
 *   [528,656) the 64 bf16 RoPE values, bit for bit. */
int oracle_dsmla_quant_write(const uint16_t* nope, const uint16_t* rope, int64_t n,
                             const int64_t* slot_mapping, uint8_t* cache,
                             int64_t num_blocks, int block_size,
                             int64_t block_stride, int64_t entry_stride)
{
    codec_init();
    const float inv448 = (float)(1.0 / 448.0);
    const float floor_scale = 1.1754944e-38f;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < n; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        if (blk >= num_blocks) { bad = 1; continue; }
        uint8_t* e = cache + blk * block_stride + off * entry_stride;
        for (int tile = 0; tile < 4; ++tile) {
            const uint16_t* src = nope + t * 512 + tile * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16_to_f32(src[i]));
                if (a > amax) amax = a;
            }
            float sc = amax * inv448;
            if (!(sc >= floor_scale)) sc = floor_scale;
            for (int i = 0; i < 128; ++i)
                e[tile * 128 + i] = oracle_e4m3_encode(bf16_to_f32(src[i]) / sc);
            memcpy(e + 512 + 4 * tile, &sc, 4);
        }
        memcpy(e + 528, rope + t * 64, 128);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Fused RMSNorm + RoPE + fp8_ds_mla write: the whole per-token step of the    */
/* page's _fused_norm_rope_kernel, fp8_ds_mla branch [DSMLA]; the norm and the */
/* rotation follow the readings listed at the top of this function             */
/* ------------------------------------------------------------------------- */

/* Nearest bf16, ties to the even bf16 (NaN stays a quiet NaN). */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* One 128-value NoPE tile of f32 values: sc = max(amax * f32(1/448),
 * 1.1754944e-38) (f32 multiply), codes = enc(y / sc) (IEEE f32 division). */
static float code_tile_f32(const float* y, uint8_t* codes)
{
    const float inv448 = (float)(1.0 / 448.0);
    const float floor_scale = 1.1754944e-38f;
    float amax = 0.0f;
    for (int i = 0; i < 128; ++i) {
        float a = fabsf(y[i]);
        if (a > amax) amax = a;
    }
    float sc = amax * inv448;
    if (!(sc >= floor_scale)) sc = floor_scale;
    for (int i = 0; i < 128; ++i) codes[i] = oracle_e4m3_encode(y[i] / sc);
    return sc;
}

/* Per token t with slot_mapping[t] >= 0 (readings of what the page leaves open):
 *   RMSNorm of the 512 bf16 NoPE values x with weights g (bf16):
 *     S = sum_i x_i^2 in double (every square of a bf16 value has at most 16
 *         significant bits, so the sum is exact for these inputs and does not
 *         depend on the order of the terms);
 *     t = (float)(S / 512.0 + (double)eps): the mean square plus eps, formed in
 *         double and rounded once to f32;
 *     r = 1 / sqrt(t) in f32 (IEEE square root, then IEEE division);
 *     y_i = (x_i * r) * g_i in f32 (two rounded products, no fused multiply-add).
 *   The 512 y are coded as the fp8_ds_mla NoPE (4 tiles of 128, as above) and
 *   the tile scales follow them.
 *   RoPE, interleaved pairs (the page stores r1, r2 at 2i, 2i+1): for pair i of
 *   the 64 bf16 values, at position p = positions[t], with c = cos_sin[p*64 + i]
 *   and s = cos_sin[p*64 + 32 + i] (the cosine half, then the sine half):
 *     r1 = x0*c - x1*s,  r2 = x0*s + x1*c  in f32 (products rounded, then the
 *     sum), each stored as bf16, nearest with ties to even.
 * A slot past the pool or a position outside [0, max_pos) skips the token and
 * makes the call return -1. */
int oracle_dsmla_norm_rope_write(const uint16_t* kv, const uint16_t* pe, const uint16_t* gamma,
                                 float eps, const int64_t* positions, const float* cos_sin,
                                 int64_t max_pos, const int64_t* slot_mapping, int64_t n,
                                 uint8_t* cache, int64_t num_blocks, int block_size,
                                 int64_t block_stride, int64_t entry_stride)
{
    codec_init();
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < n; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, off = slot % block_size;
        int64_t p = positions[t];
        if (blk >= num_blocks || p < 0 || p >= max_pos) { bad = 1; continue; }
        uint8_t* e = cache + blk * block_stride + off * entry_stride;
        const uint16_t* x = kv + t * 512;
        double S = 0.0;
        for (int i = 0; i < 512; ++i) {
            double v = (double)bf16_to_f32(x[i]);
            S += v * v;
        }
        float t32 = (float)(S / 512.0 + (double)eps);
        float r = 1.0f / sqrtf(t32);
        float y[512];
        for (int i = 0; i < 512; ++i) {
            float xr = bf16_to_f32(x[i]) * r;
            y[i] = xr * bf16_to_f32(gamma[i]);
        }
        for (int tile = 0; tile < 4; ++tile) {
            float sc = code_tile_f32(y + 128 * tile, e + 128 * tile);
            memcpy(e + 512 + 4 * tile, &sc, 4);
        }
        const uint16_t* q = pe + t * 64;
        const float* cs = cos_sin + p * 64;
        uint16_t out[64];
        for (int i = 0; i < 32; ++i) {
            float x0 = bf16_to_f32(q[2 * i]), x1 = bf16_to_f32(q[2 * i + 1]);
            float c = cs[i], s = cs[32 + i];
            float a = x0 * c, b = x1 * s, u = x0 * s, w = x1 * c;
            out[2 * i] = f32_to_bf16(a - b);
            out[2 * i + 1] = f32_to_bf16(u + w);
        }
        memcpy(e + 528, out, 128);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Query side: fused_q with quantize_mqa [DSMLA]; the indexer query and head  */
/* weights [SCORE]; the readings sit with each function                       */
/* ------------------------------------------------------------------------- */

/* n f32 values coded with one scale: s = max(amax / 448, FLT_MIN) (IEEE f32
 * division, the indexer-K rule of [SCORE]), codes = enc(x / s) (IEEE f32
 * division).  Returns s. */
static float code_vector_div448(const float* x, int n, uint8_t* codes)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f;
    if (!(s >= FLT_MIN)) s = FLT_MIN;
    for (int i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(x[i] / s);
    return s;
}

/* The MQA query of the sparse MLA attention ([DSMLA]: fused_q's quantize_mqa
 * flag selects an FP8 MQA query or the BF16 pair (ql_nope, q_pe)).  Readings of
 * what the page leaves open: per token t and head h,
 *   q_pe is rotated as the cache's RoPE values are (interleaved pairs; with
 *   p = positions[t], c = cos_sin[p*64 + i], s = cos_sin[p*64 + 32 + i]:
 *   r1 = x0*c - x1*s, r2 = x0*s + x1*c in f32, products rounded, then the sum,
 *   each stored as bf16, nearest with ties to even);
 *   quantize_mqa == 0: out_pe[t,h] = the 64 rotated bf16 values (ql_nope is
 *   returned as it came in);
 *   quantize_mqa != 0: the 576 values [ql_nope (512) | rotated q_pe (64)]
 *   (each bf16, exact in f32) coded with one scale per (token, head),
 *   s = max(amax / 448, FLT_MIN), codes = enc(v / s): out_mqa[t,h,576] and
 *   out_scale[t,h] = s.
 * A position outside [0, max_pos) skips the token and makes the call return -1. */
int oracle_fused_q(const uint16_t* ql_nope, const uint16_t* q_pe, const int64_t* positions,
                   const float* cos_sin, int64_t max_pos, int64_t tokens, int heads, int quantize_mqa,
                   uint16_t* out_pe, uint8_t* out_mqa, float* out_scale)
{
    codec_init();
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < tokens; ++t) {
        int64_t p = positions[t];
        if (p < 0 || p >= max_pos) { bad = 1; continue; }
        const float* cs = cos_sin + p * 64;
        for (int h = 0; h < heads; ++h) {
            const int64_t th = t * heads + h;
            const uint16_t* x = q_pe + th * 64;
            uint16_t rot[64];
            for (int i = 0; i < 32; ++i) {
                float x0 = bf16_to_f32(x[2 * i]), x1 = bf16_to_f32(x[2 * i + 1]);
                float c = cs[i], s = cs[32 + i];
                float a = x0 * c, b = x1 * s, u = x0 * s, w = x1 * c;
                rot[2 * i] = f32_to_bf16(a - b);
                rot[2 * i + 1] = f32_to_bf16(u + w);
            }
            if (!quantize_mqa) {
                memcpy(out_pe + th * 64, rot, 128);
                continue;
            }
            float v[576];
            for (int i = 0; i < 512; ++i) v[i] = bf16_to_f32(ql_nope[th * 512 + i]);
            for (int i = 0; i < 64; ++i) v[512 + i] = bf16_to_f32(rot[i]);
            out_scale[th] = code_vector_div448(v, 576, out_mqa + th * 576);
        }
    }
    return bad ? -1 : 0;
}

/* The indexer's FP8 query and head weights [SCORE]: per token t and head h of
 * the bf16 query q[t,h,:] (head_dim values), s = max(amax / 448, FLT_MIN),
 * q_fp8[t,h,:] = enc(q / s), w_out[t,h] = w[t,h] * s (f32 product).  Reading:
 * the score is sum_h w_h * ReLU((s_h * q_fp8_h) . k); as s_h > 0,
 * ReLU(s_h * x) = s_h * ReLU(x), so folding s_h into the weight lets the
 * logits take the fp8 codes as they are. */
int oracle_quant_q(const uint16_t* q, const float* w, int64_t tokens, int heads, int head_dim,
                   uint8_t* q_fp8, float* w_out)
{
    codec_init();
    if (head_dim > 1024) return -2;
#pragma omp parallel for schedule(static)
    for (int64_t th = 0; th < tokens * heads; ++th) {
        float v[1024];
        for (int d = 0; d < head_dim; ++d) v[d] = bf16_to_f32(q[th * head_dim + d]);
        float s = code_vector_div448(v, head_dim, q_fp8 + th * head_dim);
        w_out[th] = w[th] * s;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Sparse MLA decode attention over the fp8_ds_mla cache [DSMLA] [ATOM]       */
/* ------------------------------------------------------------------------- */

/* The consumer of the global top-k indices: for query token t and head h,
 * attention over the cache entries its index row names.  [DSMLA] gives the
 * query as the bf16 pair (ql_nope [512], q_pe [64]) and the 656-byte entry;
 * [ATOM] gives the per-query 2-D buffer of global paged-KV indices.  Neither
 * prints the attention itself; the reading is plain scaled-dot-product
 * attention over the selected entries:
 *   key j (slot g = indices[t, j] >= 0) at blk = g / bs, off = g % bs:
 *     k[i] = dec(code[i]) * scale[i / 128]   (i < 512, exact in double)
 *     k[512 + i] = rope[i]                   (bf16, exact)
 *     v = k[0 .. 512)                        (the latent is both key and value)
 *   z_j = sm_scale * (q_nope . k[0..512) + q_pe . k[512..576))
 *   out[t,h,:] = sum_j exp(z_j - m) v_j / sum_j exp(z_j - m),  m = max_j z_j
 *   lse[t,h]   = m + log(sum_j exp(z_j - m))   (natural log)
 * A negative index names no key; a row with no key has out = 0 and
 * lse = -inf.  An index past the cache is skipped and makes the call return -1.
 * Everything is in double. */
int oracle_dsmla_sparse_decode(const uint16_t* q_nope, const uint16_t* q_pe,
                               const uint8_t* cache, int64_t num_blocks, int block_size,
                               int64_t block_stride, int64_t entry_stride,
                               const int32_t* indices, int64_t tokens, int heads, int topk,
                               double sm_scale, double* out, double* lse)
{
    codec_init();
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t t = 0; t < tokens; ++t) {
        double* kd = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * 576);
        double* z = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
        int* ok = (int*)malloc(sizeof(int) * (size_t)(topk > 0 ? topk : 1));
        for (int j = 0; j < topk; ++j) {
            int64_t g = indices[t * topk + j];
            ok[j] = 0;
            if (g < 0) continue;
            if (g / block_size >= num_blocks) { bad = 1; continue; }
            const uint8_t* e = cache + (g / block_size) * block_stride + (g % block_size) * entry_stride;
            for (int i = 0; i < 512; ++i) {
                float sc;
                memcpy(&sc, e + 512 + 4 * (i / 128), 4);
                kd[(size_t)j * 576 + i] = oracle_e4m3_decode(e[i]) * (double)sc;
            }
            for (int i = 0; i < 64; ++i) {
                uint16_t r;
                memcpy(&r, e + 528 + 2 * i, 2);
                kd[(size_t)j * 576 + 512 + i] = (double)bf16_to_f32(r);
            }
            ok[j] = 1;
        }
        for (int h = 0; h < heads; ++h) {
            const uint16_t* qn = q_nope + ((size_t)t * heads + h) * 512;
            const uint16_t* qp = q_pe + ((size_t)t * heads + h) * 64;
            double m = -INFINITY;
            for (int j = 0; j < topk; ++j) {
                if (!ok[j]) continue;
                const double* k = kd + (size_t)j * 576;
                double s = 0.0;
                for (int i = 0; i < 512; ++i) s += (double)bf16_to_f32(qn[i]) * k[i];
                for (int i = 0; i < 64; ++i) s += (double)bf16_to_f32(qp[i]) * k[512 + i];
                z[j] = sm_scale * s;
                if (z[j] > m) m = z[j];
            }
            double* o = out + ((size_t)t * heads + h) * 512;
            for (int i = 0; i < 512; ++i) o[i] = 0.0;
            if (m == -INFINITY) {
                lse[(size_t)t * heads + h] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int j = 0; j < topk; ++j) {
                if (!ok[j]) continue;
                const double p = exp(z[j] - m);
                l += p;
                const double* v = kd + (size_t)j * 576;
                for (int i = 0; i < 512; ++i) o[i] += p * v[i];
            }
            for (int i = 0; i < 512; ++i) o[i] /= l;
            lse[(size_t)t * heads + h] = m + log(l);
        }
        free(kd);
        free(z);
        free(ok);
    }
    return bad ? -1 : 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
