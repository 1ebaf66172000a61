/*
 * dsix.h -- C ABI of the GB300 (sm_103a) DeepSeek-V3.2 sparse-attention
 * indexer hot path: indexer-K quantise/write, paged gather, FP8 MQA logits
 * (paged decode and contiguous prefill), per-row top-k with remap to global
 * paged-KV slots, the fp8_ds_mla cache write (alone or fused with the RMSNorm
 * and RoPE of its token), and the sparse MLA decode attention that consumes the
 * global indices.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless a
 *   comment says otherwise.  The library never allocates, frees or retains
 *   caller memory.
 * - Every call is asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *   stream).  No entry point synchronises, reads device memory on the host, or
 *   allocates, so every call can be captured into a CUDA graph (the host-sync
 *   failure that vLLM PR #36250 "[kernel] Fix FP8 paged MQA fallback for CUDA
 *   graph capture" fixes cannot occur here).  The first call of each entry
 *   point on a device sets kernel attributes; make it before any capture.
 * - Return value: IX_OK (0) or a negative IX_ERR_* code.  Argument errors are
 *   detected on the host before anything is launched; IX_ERR_CUDA reports a
 *   launch failure from the CUDA runtime.
 * - Values the host cannot see (block-table entries, lengths) are checked on
 *   the device: a kernel that meets one that is out of range skips the access
 *   and ORs a bit into a per-device status word, which ix_device_status()
 *   returns (synchronously) and clears.
 * - Supported shapes: head_dim 128, 64 heads, block_size 64 (the DeepSeek-V3.2
 *   indexer), next_n 1..2; 128 query heads for the sparse MLA decode.
 *   Anything else returns IX_ERR_UNSUPPORTED.
 * - fp8 means OCP E4M3 (bias 7, largest finite 448); conversions round to
 *   nearest even and saturate.
 *
 * Indexer-K paged cache layout (vLLM PR #25869 "[Model] Support Deepseek
 * V3.2", code review of cp_gather_indexer_k_quant_cache): uint8
 * [num_blocks][block_size*(head_dim+4)]; a block holds block_size x head_dim
 * fp8 values token by token, then block_size fp32 scales (4 bytes each).  At
 * 64 x 128 a block is 8448 bytes: token j's values at [128j, 128j+128), its
 * scale at 8192 + 4j.  The cache base must be 16-byte aligned.
 */
#ifndef DSIX_H
#define DSIX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported from the shared library; every other symbol stays hidden. */
#if defined(__GNUC__)
#define IX_API __attribute__((visibility("default")))
#else
#define IX_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* ix_stream_t;

enum {
    IX_OK = 0,
    IX_ERR_NULL = -1,         /* a required pointer is NULL */
    IX_ERR_SHAPE = -2,        /* a size or stride is negative or inconsistent */
    IX_ERR_UNSUPPORTED = -3,  /* head_dim / heads / block_size / next_n / k / ld not supported */
    IX_ERR_ALIGN = -4,        /* a base pointer or stride breaks the stated alignment */
    IX_ERR_WORKSPACE = -5,    /* workspace missing or smaller than its stated size */
    IX_ERR_CUDA = -6,         /* the CUDA runtime rejected a launch or a query */
    IX_ERR_DEVICE_CHECK = -7  /* returned by ix_device_status when a device check fired */
};

/* Bits of the device status word (see ix_device_status). */
enum {
    IX_DEV_BAD_SLOT = 1,        /* slot_mapping entry past the block pool: token skipped */
    IX_DEV_BAD_BLOCK = 2,       /* block_table entry outside [0, num_blocks): access skipped */
    IX_DEV_ROW_TOO_LONG = 4,    /* a visible row is longer than ld: columns >= ld dropped */
    IX_DEV_BAD_RANGE = 8,       /* ks/ke outside [0, tk], or cu_seq_lens past out_capacity */
    IX_DEV_TIMEOUT = 16,        /* a pipeline wait gave up (never expected) */
    IX_DEV_BAD_POSITION = 32,   /* a RoPE position outside [0, max_pos): token skipped */
    IX_DEV_BAD_HIST = 64        /* a top-k histogram did not match its row (workspace not zero before use) */
};

/* Human-readable name of a status code (static string, never NULL). */
IX_API const char* ix_status_string(int status);

/*
 * Reads and clears the calling device's status word.  SYNCHRONOUS: it waits
 * for all work on the device.  Diagnostic only -- never call it on the hot
 * path or during stream capture.  *status_out (may be NULL) receives the
 * IX_DEV_* bits; returns IX_OK if no bit was set, IX_ERR_DEVICE_CHECK if one
 * was, IX_ERR_CUDA on a runtime error.
 */
IX_API int ix_device_status(int* status_out);

/*
 * ix_quant_write_k -- quantise new indexer keys and write them into the paged
 * cache.  For every token t with slot = slot_mapping[t] >= 0:
 *   amax  = max_i |k[t,i]|                       (bf16 values, exact in f32)
 *   scale = max(amax / 448, FLT_MIN)             (IEEE f32 division)
 *   v[i]  = fp8(k[t,i] / scale)                  (IEEE f32 division, RNE, satfinite)
 * written to block slot/block_size, row slot%block_size of the layout above.
 * Tokens with a negative slot are skipped.  This is the DeepSeek-V3.2 indexer
 * K quantisation, into the layout that vLLM PR #25869's
 * cp_gather_indexer_k_quant_cache review reads back.
 *   k_bf16        bf16 [n, head_dim], row-major, 16-byte aligned
 *   slot_mapping  int64 [n]
 *   cache         uint8 [num_blocks, block_size*(head_dim+4)], 16-byte aligned
 */
IX_API int ix_quant_write_k(const void* k_bf16, int64_t n, int head_dim,
                     const int64_t* slot_mapping, uint8_t* cache,
                     int64_t num_blocks, int block_size, ix_stream_t stream);

/*
 * ix_gather_k -- copy ragged paged indexer K into contiguous buffers (vLLM PR
 * #25869, code review of cp_gather_indexer_k_quant_cache).  For each request b
 * with s = cu_seq_lens[b+1] - cu_seq_lens[b] > 0 and each i < s:
 *   out_k[cu_seq_lens[b] + i, :]   = values of row i%bs of block block_table[b, i/bs]
 *   out_scale[cu_seq_lens[b] + i]  = that row's fp32 scale
 * i.e. all full blocks, then the first s%bs rows of the last block.  Rows at or
 * past cu_seq_lens[batch] are not written.
 *   block_table   int32 [batch, bt_stride]
 *   cu_seq_lens   int32 [batch+1], non-decreasing, cu_seq_lens[0] = 0
 *   out_k         fp8 (uint8) [out_capacity, head_dim], 16-byte aligned
 *   out_scale     fp32 [out_capacity]
 *   out_capacity  host-side upper bound on cu_seq_lens[batch]; rows at or past
 *                 it are never written (IX_DEV_BAD_RANGE if that drops any)
 */
IX_API int ix_gather_k(const uint8_t* cache, int64_t num_blocks, int block_size, int head_dim,
                const int32_t* block_table, int64_t bt_stride,
                const int32_t* cu_seq_lens, int batch, uint8_t* out_k,
                float* out_scale, int64_t out_capacity, ix_stream_t stream);

/*
 * ix_paged_mqa_logits -- decode indexer logits over the paged cache (the op
 * that vLLM PR #36250's fp8_paged_mqa_logits fallback computes).  Row
 * r = b*next_n + j (j < next_n) sees L = context_lens[b] - next_n + 1 + j keys;
 * for s < L:
 *   logits[r, s] = k_scale[s] * sum_h w[r, h] * ReLU(sum_d q[b, j, h, d] * k[s, d])
 * with k and k_scale read through block_table[b, s/64].  FP8 x FP8 products,
 * FP32 accumulation (tcgen05 tensor cores).  With clean_logits != 0 the
 * entries [L, ld) are set to -inf; with 0 they are left untouched (the
 * clean_logits=False mode discussed in the same PR's review).
 *   q_fp8         uint8 (e4m3) [batch, next_n, heads, head_dim], 16-byte aligned
 *   w             fp32 [batch*next_n, heads], 16-byte aligned
 *   context_lens  int32 [batch]
 *   block_table   int32 [batch, bt_stride]
 *   logits        fp32 [batch*next_n, ld]; ld >= every L, ld % 4 == 0
 */
IX_API int ix_paged_mqa_logits(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                        int64_t num_blocks, int block_size,
                        const int32_t* context_lens, const int32_t* block_table,
                        int64_t bt_stride, int batch, int next_n, int heads,
                        int head_dim, float* logits, int64_t ld, int clean_logits,
                        ix_stream_t stream);

/*
 * ix_mqa_logits -- prefill indexer logits over contiguous K (the dense
 * contraction that follows the gather of vLLM PR #25869).  Row t sees keys
 * [ks[t], ke[t]); for j < ke[t] - ks[t]:
 *   logits[t, j] = k_scale[ks[t]+j] * sum_h w[t, h] * ReLU(q[t, h, :] . k[ks[t]+j, :])
 * Column j is the request-local key index when ks[t] is the request's first
 * gathered row.  clean_logits as above, for [ke[t]-ks[t], ld).
 *   q_fp8    uint8 (e4m3) [tq, heads, head_dim], 16-byte aligned
 *   w        fp32 [tq, heads], 16-byte aligned
 *   k_fp8    uint8 (e4m3) [tk, head_dim], 16-byte aligned
 *   k_scale  fp32 [tk], 16-byte aligned
 *   ks, ke   int32 [tq], 0 <= ks <= ke <= tk
 *   logits   fp32 [tq, ld]; ld >= every ke - ks, ld % 4 == 0
 */
IX_API int ix_mqa_logits(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                  const float* k_scale, const int32_t* ks, const int32_t* ke,
                  int64_t tq, int64_t tk, int heads, int head_dim, float* logits,
                  int64_t ld, int clean_logits, ix_stream_t stream);

/*
 * ix_topk_to_global -- per-row top-k of the indexer logits and remap of each
 * selected request-local index to its global paged-KV slot (ROCm/ATOM PR #1094
 * "[Feat] Support DSv3.2 with sglang-ATOM plugin and sglang sparse MLA",
 * Technical Details: a 2-D top-k index buffer; request-local top-k indices
 * converted to global paged KV indices).  Row r, L = row_len[r] (clamped to
 * [0, ld]), b = row_req[r]:
 *   select the min(k, L) columns s < L with the largest logits[r, s]; equal
 *   values go to the lower index; -0.0 equals +0.0;
 *   out_local[r, :]  = the selected s in ascending order, then -1 up to k
 *   out_global[r, i] = block_table[b, s/block_size]*block_size + s%block_size,
 *                      or -1 where out_local is -1
 * Logits at or past L are never read.  NaN logits give an unspecified
 * selection.
 *   logits      fp32 [rows, ld], 16-byte aligned, ld % 4 == 0
 *   row_len, row_req  int32 [rows]
 *   block_table int32 [*, bt_stride]
 *   out_local   int32 [rows, k] or NULL
 *   out_global  int32 [rows, k]
 * Supports ld <= 262144 (longer rows return IX_ERR_UNSUPPORTED) and k >= 1.
 */
IX_API int ix_topk_to_global(const float* logits, int64_t ld, int64_t rows,
                      const int32_t* row_len, const int32_t* row_req,
                      const int32_t* block_table, int64_t bt_stride, int block_size,
                      int k, int32_t* out_local, int32_t* out_global,
                      ix_stream_t stream);

/*
 * Fused logits + top-k.  The two entry points below compute exactly what
 * ix_paged_mqa_logits / ix_mqa_logits (with clean_logits = 0) followed by
 * ix_topk_to_global compute -- the same logits, the same selection, the same
 * remap -- for the rows those logits kernels produce, in one call that never
 * re-reads a row from the start for the first radix pass: while the logits
 * kernel writes a row with more than k visible keys, it also counts the first
 * radix digit of each logit (the top 11 bits of its order key) into the row's
 * histogram, and the selection that follows starts from the digit that holds
 * the k-th largest key.  This is the clean_logits=False mode of vLLM PR #36250
 * "[kernel] Fix FP8 paged MQA fallback for CUDA graph capture" (review thread:
 * the logits past each row's end need no -inf fill, since the selection never
 * reads them) feeding the 2-D top-k index buffer of ROCm/ATOM PR #1094
 * "[Feat] Support DSv3.2 with sglang-ATOM plugin and sglang sparse MLA"
 * (Technical Details: request-local top-k indices converted to global paged KV
 * indices).
 *
 * Workspace: ix_topk_hist_workspace_size(rows) bytes (8448 per row: 64 coarse
 * and 2048 fine u32 bins), 16-byte aligned, owned by the caller.  It must be
 * ALL ZERO before its first use; every call that completes leaves it all zero
 * again, so set it to zero once when it is allocated.  Calls that share a
 * workspace must not overlap on the GPU.  If a call stops short (a pipeline
 * wait gives up: IX_DEV_TIMEOUT), clear the workspace before reusing it.  A
 * histogram that does not match its row (a workspace that was not zero) sets
 * IX_DEV_BAD_HIST; that row's output is then incomplete and padded with -1.
 * `logits` is written as by the unfused call (entries past each row's length
 * are left untouched) and is read back by the selection.
 */
IX_API size_t ix_topk_hist_workspace_size(int64_t rows);

/*
 * ix_paged_mqa_logits_topk -- ix_paged_mqa_logits (clean_logits = 0) and then
 * ix_topk_to_global over its rows: row r = b*next_n + j has length
 * L = clamp(context_lens[b] - next_n + 1 + j, 0, ld) and request b; its indices
 * are remapped through block_table[b, :] with block_size (64).  Arguments as
 * in those two calls; out_local may be NULL.  Errors, before any launch: those
 * of ix_paged_mqa_logits; IX_ERR_UNSUPPORTED for k < 1 or ld > 262144;
 * IX_ERR_WORKSPACE for a missing or small workspace; IX_ERR_ALIGN for a
 * workspace that is not 16-byte aligned; IX_ERR_NULL for out_global.
 */
IX_API int ix_paged_mqa_logits_topk(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                        int64_t num_blocks, int block_size, const int32_t* context_lens,
                        const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                        int heads, int head_dim, float* logits, int64_t ld, int k,
                        int32_t* out_local, int32_t* out_global, void* workspace,
                        size_t workspace_bytes, ix_stream_t stream);

/*
 * ix_mqa_logits_topk -- ix_mqa_logits (clean_logits = 0) and then
 * ix_topk_to_global over its rows: row t has length L = ke[t] - ks[t] (clamped
 * as ix_mqa_logits clamps it, and to ld) and request row_req[t]; column j is
 * remapped through block_table[row_req[t], j / block_size] (j is the
 * request-local key index when ks[t] is the request's first gathered row).
 * Arguments as in those two calls; row_req int32 [tq]; out_local may be NULL.
 * Errors, before any launch: those of ix_mqa_logits; the k / ld / workspace
 * errors of ix_paged_mqa_logits_topk; IX_ERR_SHAPE for bt_stride < 0;
 * IX_ERR_UNSUPPORTED for block_size < 1; IX_ERR_NULL for row_req, block_table
 * or out_global.
 */
IX_API int ix_mqa_logits_topk(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                        const float* k_scale, const int32_t* ks, const int32_t* ke, int64_t tq,
                        int64_t tk, int heads, int head_dim, float* logits, int64_t ld,
                        const int32_t* row_req, const int32_t* block_table, int64_t bt_stride,
                        int block_size, int k, int32_t* out_local, int32_t* out_global,
                        void* workspace, size_t workspace_bytes, ix_stream_t stream);

/*
 * The two halves of the fused calls, for callers that place the selection
 * themselves (another stream, a later point of a graph) or time the halves:
 * ix_*_logits_hist runs the logits kernel of the fused call (logits as
 * ix_*_logits with clean_logits = 0, plus the histograms of the rows with
 * more than k keys), ix_topk_from_hist the selection.  Between them the
 * workspace holds the histograms: ix_topk_from_hist must follow on the same
 * rows, with row_len[r] equal to the length the logits call gave row r (the
 * clamped L above) and the same k, and it leaves the workspace zero again.
 * Errors as in the fused calls (ix_topk_from_hist: those of
 * ix_topk_to_global, then the workspace errors).
 */
IX_API int ix_paged_mqa_logits_hist(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                        int64_t num_blocks, int block_size, const int32_t* context_lens,
                        const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                        int heads, int head_dim, float* logits, int64_t ld, int k,
                        void* workspace, size_t workspace_bytes, ix_stream_t stream);
IX_API int ix_mqa_logits_hist(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                        const float* k_scale, const int32_t* ks, const int32_t* ke, int64_t tq,
                        int64_t tk, int heads, int head_dim, float* logits, int64_t ld, int k,
                        void* workspace, size_t workspace_bytes, ix_stream_t stream);
IX_API int ix_topk_from_hist(const float* logits, int64_t ld, int64_t rows,
                        const int32_t* row_len, const int32_t* row_req,
                        const int32_t* block_table, int64_t bt_stride, int block_size, int k,
                        int32_t* out_local, int32_t* out_global, void* workspace,
                        size_t workspace_bytes, ix_stream_t stream);

/*
 * dsmla_quant_write -- the fp8_ds_mla cache write (vLLM PR #47090, prhub
 * summary, key source snippet of _fused_norm_rope_kernel, fp8_ds_mla branch).
 * For every token t with slot = slot_mapping[t] >= 0, at byte
 * (slot/block_size)*block_stride_bytes + (slot%block_size)*entry_stride_bytes:
 *   bytes [0,512)    fp8 NoPE: for tile c of 128 values,
 *                    sc_c = max(amax_c * f32(1/448), 1.1754944e-38) (f32 multiply),
 *                    v = fp8(x / sc_c) (IEEE f32 division, RNE, satfinite)
 *   bytes [512,528)  sc_0..sc_3 as fp32
 *   bytes [528,656)  the 64 bf16 RoPE values, copied bit for bit
 * Tokens with a negative slot are skipped.  The RoPE values arrive already
 * rotated (normalisation and rotation are the caller's).
 *   nope_bf16  bf16 [n, 512], 16-byte aligned;  rope_bf16  bf16 [n, 64], 16-byte aligned
 *   cache      uint8, 16-byte aligned; block_stride_bytes and entry_stride_bytes
 *              multiples of 16, entry_stride_bytes >= 656
 */
IX_API int dsmla_quant_write(const void* nope_bf16, const void* rope_bf16, int64_t n,
                      const int64_t* slot_mapping, uint8_t* cache, int64_t num_blocks,
                      int block_size, int64_t block_stride_bytes,
                      int64_t entry_stride_bytes, ix_stream_t stream);

/*
 * dsmla_norm_rope_write -- the whole per-token step that the fp8_ds_mla write
 * above is the last part of (vLLM PR #47090, prhub summary: the fp8_ds_mla
 * branch of _fused_norm_rope_kernel writes the normalised KV and the rotated
 * RoPE values).  The page prints neither the norm nor the rotation; this entry
 * point computes, for every token t with slot = slot_mapping[t] >= 0:
 *   RMSNorm of the 512 NoPE values x with weights g:
 *     S = sum x_i^2, exact and rounded once to double (each square of a bf16
 *     value has at most 16 significant bits; squares more than 2^38 below the
 *     token's largest are cut to a multiple of 2^-38 of it),
 *     t = f32(S / 512 + eps), r = 1 / sqrt(t) (f32: IEEE square root, then
 *     IEEE division), y_i = (x_i * r) * g_i (f32, two rounded products);
 *   the 512 y coded as dsmla_quant_write codes its NoPE values (tiles of 128,
 *   sc = max(amax * f32(1/448), 1.1754944e-38), v = fp8(y / sc)), the tile
 *   scales after them;
 *   RoPE on interleaved pairs: with p = positions[t], for pair i (values 2i,
 *   2i + 1) c = cos_sin[p*64 + i], s = cos_sin[p*64 + 32 + i],
 *     r1 = x0*c - x1*s, r2 = x0*s + x1*c (f32: products rounded, then the sum),
 *   stored as bf16 (nearest, ties to even) at 2i and 2i + 1 of bytes [528,656).
 * Tokens with a negative slot are skipped; a slot past the pool sets
 * IX_DEV_BAD_SLOT and a position outside [0, max_pos) sets IX_DEV_BAD_POSITION,
 * and the token is skipped.
 *   kv_bf16     bf16 [n, 512], 16-byte aligned (the compressed KV before the norm)
 *   pe_bf16     bf16 [n, 64], 4-byte aligned (the RoPE part before the rotation)
 *   gamma_bf16  bf16 [512], 16-byte aligned (the norm weights)
 *   positions   int64 [n];  cos_sin  f32 [max_pos, 64] (32 cosines, then 32 sines)
 *   cache, strides: as dsmla_quant_write
 */
IX_API int dsmla_norm_rope_write(const void* kv_bf16, const void* pe_bf16, const void* gamma_bf16,
                      float eps, const int64_t* positions, const float* cos_sin,
                      int64_t max_pos, const int64_t* slot_mapping, int64_t n,
                      uint8_t* cache, int64_t num_blocks, int block_size,
                      int64_t block_stride_bytes, int64_t entry_stride_bytes,
                      ix_stream_t stream);

/*
 * dsmla_sparse_decode -- sparse MLA decode attention, the consumer of the
 * global top-k indices (vLLM PR #47090, prhub summary: the FlashMLA sparse path
 * takes the bf16 query pair (ql_nope, q_pe) and the fp8_ds_mla cache; ROCm/ATOM
 * PR #1094, Technical Details: a per-query buffer of global paged-KV indices).
 * The pages print no attention formula; this entry point computes plain
 * softmax attention over the selected entries.  For token t and head h, with
 * the entry of slot g = indices[t*topk + j] >= 0 at
 * cache + (g / block_size) * block_stride_bytes + (g % block_size) * entry_stride_bytes:
 *   k[i] = e4m3(code[i]) * scale[i / 128]  (i < 512),  k[512 + i] = rope[i],
 *   v = k[0, 512),  z_j = sm_scale * (q_nope[t,h] . k[0,512) + q_pe[t,h] . k[512,576)),
 *   out[t,h,:] = sum_j exp(z_j - m) v_j / sum_j exp(z_j - m),  m = max_j z_j,
 *   lse[t,h] = m + ln(sum_j exp(z_j - m)).
 * A negative index names no key; a token with no key gets out = 0 and
 * lse = -inf.  An index past the pool sets IX_DEV_BAD_SLOT and is treated as
 * none.  Duplicate indices count once each.
 * Arithmetic: keys and values are dequantised to bf16 (f32 product, then
 * nearest-even), both products run on the tensor cores in bf16 with f32
 * accumulation, the softmax weights are rounded to bf16, the output to bf16.
 *   q_nope_bf16  bf16 [tokens, heads, 512], contiguous, 16-byte aligned
 *   q_pe_bf16    bf16 [tokens, heads, 64], contiguous, 16-byte aligned
 *   cache        fp8_ds_mla entries (see dsmla_quant_write), 16-byte aligned;
 *                block_stride_bytes and entry_stride_bytes multiples of 16,
 *                entry_stride_bytes >= 656, block_stride_bytes >=
 *                block_size * entry_stride_bytes
 *   indices      int32 [tokens, topk] global slots (-1: none)
 *   heads        must be 128;  1 <= topk <= 65536;  sm_scale > 0 and finite
 *   out_bf16     bf16 [tokens, heads, 512], 16-byte aligned (written)
 *   lse          f32 [tokens, heads] (written)
 *   workspace    16-byte aligned device scratch of at least
 *                dsmla_sparse_decode_workspace_size(tokens, heads, topk) bytes
 *                (per split of 256 indices: its normalised output and lse);
 *                IX_ERR_WORKSPACE if missing or smaller.  Owned by the caller,
 *                in use until the call's work on `stream` completes.
 * Errors, checked on the host in this order before anything is launched:
 *   IX_ERR_SHAPE        tokens, num_blocks, a stride or topk negative
 *   IX_ERR_UNSUPPORTED  heads != 128, block_size < 1, topk outside [1, 65536],
 *                       sm_scale not positive and finite
 *   IX_OK               tokens == 0 (nothing is read or written)
 *   IX_ERR_NULL         a pointer is NULL (cache may be NULL when num_blocks == 0)
 *   IX_ERR_SHAPE        entry_stride_bytes < 656 or block_stride_bytes <
 *                       block_size * entry_stride_bytes
 *   IX_ERR_ALIGN        a base or stride breaks the alignment above (indices and
 *                       lse need 4 bytes)
 *   IX_ERR_UNSUPPORTED  tokens * 128 or tokens * ceil(topk / 256) above INT32_MAX
 *   IX_ERR_WORKSPACE    workspace NULL or smaller than its size
 *   IX_ERR_ALIGN        workspace not 16-byte aligned
 *   IX_ERR_CUDA         the tensor-map encoder or a launch failed
 * dsmla_sparse_decode_workspace_size returns 0 when tokens, heads or topk is
 * not positive.  If a pipeline wait gives up (IX_DEV_TIMEOUT in the device
 * status word, never expected), the splits it cut short are left out of the
 * merge, so out and lse are then incomplete.
 */
IX_API size_t dsmla_sparse_decode_workspace_size(int64_t tokens, int heads, int topk);
IX_API int dsmla_sparse_decode(const void* q_nope_bf16, const void* q_pe_bf16, const uint8_t* cache,
                    int64_t num_blocks, int block_size, int64_t block_stride_bytes,
                    int64_t entry_stride_bytes, const int32_t* indices, int64_t tokens,
                    int heads, int topk, float sm_scale, void* out_bf16, float* lse,
                    void* workspace, size_t workspace_bytes, ix_stream_t stream);

/*
 * dsmla_sparse_decode_noalloc -- dsmla_sparse_decode without a caller
 * workspace: the split outputs go to scratch the library holds in a file-scope
 * device array (128 (token, split) pairs: tokens * ceil(topk / 256) <= 128,
 * e.g. 16 tokens at topk 2048), placed once when the library's module loads.
 * Nothing is allocated by the call.  Same arguments and results as
 * dsmla_sparse_decode otherwise.  Its host checks are dsmla_sparse_decode's,
 * in the same order, with the capacity check in place of the workspace check:
 * a call past the scratch returns IX_ERR_WORKSPACE only when every earlier
 * check passed, and before anything is launched.  The scratch's device address
 * is looked up on the first call on a device (and again whenever the device's
 * context has changed, e.g. after a reset); make that first call before any
 * stream capture.  The scratch is shared: calls on one device must not run
 * concurrently (calls on one stream never do).
 */
IX_API int dsmla_sparse_decode_noalloc(const void* q_nope_bf16, const void* q_pe_bf16, const uint8_t* cache,
                    int64_t num_blocks, int block_size, int64_t block_stride_bytes,
                    int64_t entry_stride_bytes, const int32_t* indices, int64_t tokens,
                    int heads, int topk, float sm_scale, void* out_bf16, float* lse,
                    ix_stream_t stream);

/*
 * dsmla_fused_q -- the MQA query of the sparse MLA attention (vLLM PR #47090,
 * prhub summary: fused_q gains a quantize_mqa flag that selects an FP8 MQA
 * query or returns the BF16 pair (ql_nope, q_pe)).  The page prints no formula;
 * this entry point computes, for token t and head h (tokens x heads rows):
 *   q_pe rotated as dsmla_norm_rope_write rotates the cache's RoPE values
 *   (interleaved pairs; p = positions[t], c = cos_sin[p*64 + i],
 *   s = cos_sin[p*64 + 32 + i]; r1 = x0*c - x1*s, r2 = x0*s + x1*c in f32,
 *   products rounded, then the sum; bf16 nearest-even);
 *   quantize_mqa == 0: out_pe[t,h,:] = the 64 rotated bf16 values (the pair
 *   handed on is (ql_nope, out_pe); ql_nope is not read);
 *   quantize_mqa != 0: the 576 values v = [ql_nope[t,h,:] | rotated q_pe],
 *   coded with one scale per (token, head): sc = max(amax(|v|) / 448, FLT_MIN)
 *   (IEEE f32 division), out_mqa[t,h,i] = fp8(v[i] / sc) (IEEE f32 division,
 *   RNE, satfinite), out_scale[t,h] = sc (out_pe is not written).
 * A position outside [0, max_pos) sets IX_DEV_BAD_POSITION and the token is
 * skipped.
 *   ql_nope_bf16  bf16 [tokens, heads, 512], 16-byte aligned (quantize_mqa only)
 *   q_pe_bf16     bf16 [tokens, heads, 64], 4-byte aligned
 *   positions     int64 [tokens];  cos_sin  f32 [max_pos, 64] (32 cosines, then 32 sines)
 *   out_pe_bf16   bf16 [tokens, heads, 64], 4-byte aligned (quantize_mqa == 0)
 *   out_mqa_fp8   fp8 [tokens, heads, 576], 16-byte aligned; out_mqa_scale f32
 *                 [tokens, heads] (quantize_mqa != 0)
 * heads >= 1 (128 for DeepSeek-V3.2); IX_ERR_NULL / IX_ERR_ALIGN for the
 * buffers the chosen mode reads or writes.
 */
IX_API int dsmla_fused_q(const void* ql_nope_bf16, const void* q_pe_bf16, const int64_t* positions,
                    const float* cos_sin, int64_t max_pos, int64_t tokens, int heads, int quantize_mqa,
                    void* out_pe_bf16, uint8_t* out_mqa_fp8, float* out_mqa_scale, ix_stream_t stream);

/*
 * ix_quant_q -- the indexer's FP8 query and head weights, as the logits entry
 * points consume them (the indexer score sums w[t,h] * ReLU(q[t,h] . k) with an
 * fp8 q).  For token t and head h of the bf16 query (head_dim 128):
 *   sc = max(amax(|q[t,h,:]|) / 448, FLT_MIN) (IEEE f32 division),
 *   q_fp8[t,h,d] = fp8(q[t,h,d] / sc) (IEEE f32 division, RNE, satfinite),
 *   w_out[t,h] = w[t,h] * sc (f32 product).
 * Because sc > 0, ReLU(sc * x) = sc * ReLU(x): the logits of (q_fp8, w_out) are
 * the logits of the dequantised query sc * q_fp8 with the weight w.
 *   q_bf16  bf16 [tokens, heads, 128], 16-byte aligned;  w, w_out f32 [tokens, heads]
 *   q_fp8   fp8 [tokens, heads, 128], 8-byte aligned
 * heads >= 1 (64 for the indexer); head_dim != 128 returns IX_ERR_UNSUPPORTED.
 */
IX_API int ix_quant_q(const void* q_bf16, const float* w, int64_t tokens, int heads, int head_dim,
                 uint8_t* q_fp8, float* w_out, ix_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSIX_H */
