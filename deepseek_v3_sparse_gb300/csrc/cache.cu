// cache.cu -- the bandwidth kernels around the caches:
//   ix_quant_write_k       indexer-K quantise + paged write
//   ix_gather_k            ragged paged gather into contiguous K
//   dsmla_quant_write      the 656-byte fp8_ds_mla entry write
//   dsmla_norm_rope_write  RMSNorm + RoPE + that entry write, fused per token
//
// All are pure streaming kernels (16-byte vector loads, grid sized to a
// multiple of the SM count); their bound is HBM bandwidth.
#include <float.h>

#include "common.cuh"

namespace dsix {
namespace {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 64;
constexpr int kBlockBytes = kBlockSize * (kHeadDim + 4);  // 8448
constexpr int kScaleOffset = kBlockSize * kHeadDim;      // 8192

__device__ __forceinline__ void unpack8(const uint4& v, float (&x)[8]) {
    x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x);
    x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
    x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z);
    x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float amax8(const float (&x)[8]) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
    return a;
}

// x[i] / scale, correctly rounded, then e4m3 (RNE, satfinite); 8 codes packed
// little-endian into two words.
__device__ __forceinline__ uint2 quant8(const float (&x)[8], float scale) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = cvt_e4m3x2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// ---------------------------------------------------------------------------
// ix_quant_write_k: one 16-lane half-warp per token, 8 bf16 (16 B) per lane.
// Loop trip counts are uniform per warp so the width-16 shuffles always see
// all 32 lanes.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_write_k_kernel(const uint4* __restrict__ k, int64_t n,
                                                            const int64_t* __restrict__ slots,
                                                            uint8_t* __restrict__ cache,
                                                            int64_t num_blocks, int* status) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         2 * wi < n; wi += warps) {
        const int64_t tok = 2 * wi + (lane >> 4);
        const bool valid = tok < n;
        float x[8];
        int64_t slot = -1;
        if (valid) {
            slot = __ldg(slots + tok);
            unpack8(__ldg(k + tok * (kHeadDim / 8) + sub), x);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
        float amax = amax8(x);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 16));
        const float scale = fmaxf(__fdiv_rn(amax, 448.0f), FLT_MIN);
        const uint2 codes = quant8(x, scale);
        if (valid && slot >= 0) {
            const int64_t blk = slot / kBlockSize;
            const int off = static_cast<int>(slot % kBlockSize);
            if (blk >= num_blocks) {
                if (sub == 0) flag(status, IX_DEV_BAD_SLOT);
            } else {
                uint8_t* base = cache + blk * kBlockBytes;
                *reinterpret_cast<uint2*>(base + off * kHeadDim + sub * 8) = codes;
                if (sub == 0) *reinterpret_cast<float*>(base + kScaleOffset + 4 * off) = scale;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// ix_gather_k: 8 lanes per token (8 x 16 B = one 128-byte row), token ->
// request by binary search over cu_seq_lens (staged in shared memory).
// ---------------------------------------------------------------------------
constexpr int kGatherSmemCu = 4096;

__global__ void __launch_bounds__(256) gather_k_kernel(const uint8_t* __restrict__ cache,
                                                       int64_t num_blocks,
                                                       const int32_t* __restrict__ bt,
                                                       int64_t bt_stride,
                                                       const int32_t* __restrict__ cu, int batch,
                                                       uint8_t* __restrict__ out_k,
                                                       float* __restrict__ out_scale,
                                                       int64_t capacity, int* status) {
    __shared__ int32_t s_cu[kGatherSmemCu];
    const bool staged = batch + 1 <= kGatherSmemCu;
    if (staged)
        for (int i = threadIdx.x; i <= batch; i += blockDim.x) s_cu[i] = __ldg(cu + i);
    __syncthreads();
    const int32_t* c = staged ? s_cu : cu;
    const int64_t total = c[batch];
    if (blockIdx.x == 0 && threadIdx.x == 0 && total > capacity) flag(status, IX_DEV_BAD_RANGE);
    const int64_t limit = total < capacity ? total : capacity;
    const int sub = threadIdx.x & 7;
    const int64_t groups = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 3;
    for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; t < limit;
         t += groups) {
        // largest b in [0, batch) with cu[b] <= t (this skips empty requests)
        int lo = 0, hi = batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (c[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int64_t i = t - c[lo];
        const int64_t blk = __ldg(bt + lo * bt_stride + i / kBlockSize);
        if (blk < 0 || blk >= num_blocks) {
            if (sub == 0) flag(status, IX_DEV_BAD_BLOCK);
            continue;
        }
        const uint8_t* src = cache + blk * kBlockBytes;
        const int off = static_cast<int>(i % kBlockSize);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + off * kHeadDim) + sub);
        reinterpret_cast<uint4*>(out_k + t * kHeadDim)[sub] = v;
        if (sub == 0) out_scale[t] = __ldg(reinterpret_cast<const float*>(src + kScaleOffset) + off);
    }
}

// ---------------------------------------------------------------------------
// dsmla_quant_write: two warps per token; a warp covers 2 tiles of 128 NoPE
// values (16 lanes x 8 values per tile).
// ---------------------------------------------------------------------------
constexpr float kInv448 = 0x1.24924ap-9f;      // f32(1/448)
constexpr float kScaleFloor = 1.1754944e-38f;  // rounds to FLT_MIN as an f32

__global__ void __launch_bounds__(256) dsmla_write_kernel(const uint4* __restrict__ nope,
                                                          const uint4* __restrict__ rope, int64_t n,
                                                          const int64_t* __restrict__ slots,
                                                          uint8_t* __restrict__ cache,
                                                          int64_t num_blocks, int block_size,
                                                          int64_t block_stride, int64_t entry_stride,
                                                          int* status) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 15;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t wi = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < 2 * n;
         wi += warps) {
        const int64_t tok = wi >> 1;
        const int half = static_cast<int>(wi & 1);
        const int tile = 2 * half + (lane >> 4);
        const int64_t slot = __ldg(slots + tok);
        if (slot < 0) continue;  // uniform across the warp
        const int64_t blk = slot / block_size;
        if (blk >= num_blocks) {
            if (lane == 0 && half == 0) flag(status, IX_DEV_BAD_SLOT);
            continue;
        }
        uint8_t* e = cache + blk * block_stride + (slot % block_size) * entry_stride;
        float x[8];
        unpack8(__ldg(nope + tok * 64 + tile * 16 + sub), x);
        float amax = amax8(x);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 16));
        const float sc = fmaxf(amax * kInv448, kScaleFloor);
        *reinterpret_cast<uint2*>(e + tile * 128 + sub * 8) = quant8(x, sc);
        if (sub == 0) *reinterpret_cast<float*>(e + 512 + 4 * tile) = sc;
        if (half == 0 && lane < 8)
            reinterpret_cast<uint4*>(e + 528)[lane] = __ldg(rope + tok * 8 + lane);
    }
}

// ---------------------------------------------------------------------------
// dsmla_norm_rope_write: one warp per token.  Lane l holds NoPE values
// [16 l, 16 l + 16) (tile l / 8) and RoPE pair l.
//   RMSNorm: S = sum x_i^2 is formed exactly in integers (below); t = f32(S / 512
//   + eps) in double, r = 1 / sqrt(t) in f32 (IEEE square root and division);
//   y = (x * r) * g in f32 with round-to-nearest products (no fused
//   multiply-add), then the ds_mla tile coding.
//   Exact S without the (slow) FP64 pipe: a bf16 value is M * 2^E with M an
//   8-bit integer, so x^2 = M^2 * 2^(2E) with M^2 < 2^16.  With Emax the
//   largest E of the token, every square is an integer multiple of 2^L,
//   L = 2 Emax - 39, as long as E >= Emax - 19; those multiples are below 2^55
//   and 512 of them sum below 2^64 in a uint64.  The sum is exact, and S =
//   double(sum) * 2^L is the exact S rounded once to double.  Squares of values
//   more than 2^19 below the token's largest are cut to their multiple of 2^L
//   (a change below 2^-38 of the largest square).
//   RoPE: r1 = x0 c - x1 s, r2 = x0 s + x1 c in f32 (products rounded, then
//   the sum), packed to bf16 with round-to-nearest-even, stored at 2l, 2l + 1.
// ---------------------------------------------------------------------------
// bf16 bits -> (M, E) with |x| = M * 2^E (M = 0 for a zero)
__device__ __forceinline__ void bf16_split(uint32_t b, uint32_t& m, int& e) {
    const uint32_t ef = (b >> 7) & 0xFFu, mf = b & 0x7Fu;
    m = ef ? (128u | mf) : mf;
    e = ef ? static_cast<int>(ef) - 134 : -133;
}

__global__ void __launch_bounds__(256, 4) dsmla_norm_rope_kernel(
    const uint4* __restrict__ kv, const uint32_t* __restrict__ pe, const uint4* __restrict__ gamma,
    float eps, const int64_t* __restrict__ positions, const float* __restrict__ cos_sin,
    int64_t max_pos, const int64_t* __restrict__ slots, int64_t n, uint8_t* __restrict__ cache,
    int64_t num_blocks, int block_size, int64_t block_stride, int64_t entry_stride, int* status) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // this lane's 16 norm weights stay in registers for every token
    float g[16];
    {
        float a[8], b[8];
        unpack8(__ldg(gamma + 2 * lane), a);
        unpack8(__ldg(gamma + 2 * lane + 1), b);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            g[i] = a[i];
            g[8 + i] = b[i];
        }
    }
    for (int64_t tok = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; tok < n;
         tok += warps) {
        // every load that depends only on the token goes out first; the
        // rotary table row follows once the position has arrived
        const int64_t slot = __ldg(slots + tok);
        const int64_t pos = __ldg(positions + tok);
        const uint4 kva = __ldg(kv + tok * 64 + 2 * lane);
        const uint4 kvb = __ldg(kv + tok * 64 + 2 * lane + 1);
        const uint32_t pair = __ldg(pe + tok * 32 + lane);
        if (slot < 0) continue;  // uniform across the warp
        const int64_t blk = slot / block_size;
        if (blk >= num_blocks || pos < 0 || pos >= max_pos) {
            if (lane == 0) flag(status, blk >= num_blocks ? IX_DEV_BAD_SLOT : IX_DEV_BAD_POSITION);
            continue;
        }
        uint8_t* e = cache + blk * block_stride + (slot % block_size) * entry_stride;
        float x[16];
        {
            float a[8], b[8];
            unpack8(kva, a);
            unpack8(kvb, b);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                x[i] = a[i];
                x[8 + i] = b[i];
            }
        }
        const float c = __ldg(cos_sin + pos * 64 + lane);
        const float sn = __ldg(cos_sin + pos * 64 + 32 + lane);
        // exact sum of squares (see above); (M, E) are recomputed in the second
        // loop rather than held, to keep the registers for more resident warps
        int emax = -1000;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t m;
            int ex;
            bf16_split(__float_as_uint(x[i]) >> 16, m, ex);
            if (m) emax = max(emax, ex);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
        double S = 0.0;
        if (emax > -1000) {  // not an all-zero token (uniform across the warp)
            const int L = 2 * emax - 39;  // every shift below is at most 39
            unsigned long long acc = 0ull;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint32_t m;
                int ex;
                bf16_split(__float_as_uint(x[i]) >> 16, m, ex);
                const unsigned long long sq = static_cast<unsigned long long>(m * m);
                const int sh = 2 * ex - L;
                acc += sh >= 0 ? (sq << sh) : (sh > -64 ? (sq >> -sh) : 0ull);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            // 2^L is a normal double for every bf16 exponent (L in [-305, 201])
            S = __dmul_rn(__ull2double_rn(acc), __longlong_as_double(static_cast<long long>(L + 1023) << 52));
        }
        const float t = __double2float_rn(__dadd_rn(__dmul_rn(S, 0x1p-9), static_cast<double>(eps)));
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(t));
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            x[i] = __fmul_rn(__fmul_rn(x[i], r), g[i]);
            amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o, 8));
        const float sc = fmaxf(__fmul_rn(amax, kInv448), kScaleFloor);
        float lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo[i] = x[i];
            hi[i] = x[8 + i];
        }
        const uint2 c0 = quant8(lo, sc), c1 = quant8(hi, sc);
        *reinterpret_cast<uint4*>(e + 16 * lane) = make_uint4(c0.x, c0.y, c1.x, c1.y);
        if ((lane & 7) == 0) *reinterpret_cast<float*>(e + 512 + 4 * (lane >> 3)) = sc;
        const float x0 = bf16_lo(pair), x1 = bf16_hi(pair);
        const float r1 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, sn));
        const float r2 = __fadd_rn(__fmul_rn(x0, sn), __fmul_rn(x1, c));
        uint32_t packed;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed) : "f"(r2), "f"(r1));  // r1 in the low half
        reinterpret_cast<uint32_t*>(e + 528)[lane] = packed;
    }
}

int grid_for(int64_t work_items, int items_per_block) {
    const int sms = num_sms();
    int64_t blocks = (work_items + items_per_block - 1) / items_per_block;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 16;
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace
}  // namespace dsix

using namespace dsix;

extern "C" int ix_quant_write_k(const void* k_bf16, int64_t n, int head_dim,
                                const int64_t* slot_mapping, uint8_t* cache, int64_t num_blocks,
                                int block_size, ix_stream_t stream) {
    if (n < 0 || num_blocks < 0) return IX_ERR_SHAPE;
    if (head_dim != kHeadDim || block_size != kBlockSize) return IX_ERR_UNSUPPORTED;
    if (n == 0) return IX_OK;
    if (!k_bf16 || !slot_mapping || !cache) return IX_ERR_NULL;
    if (!aligned16(k_bf16) || !aligned16(cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
        return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    quant_write_k_kernel<<<grid_for(n, 16), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_bf16), n, slot_mapping, cache, num_blocks, st);
    return launch_status();
}

extern "C" int ix_gather_k(const uint8_t* cache, int64_t num_blocks, int block_size, int head_dim,
                           const int32_t* block_table, int64_t bt_stride,
                           const int32_t* cu_seq_lens, int batch, uint8_t* out_k, float* out_scale,
                           int64_t out_capacity, ix_stream_t stream) {
    if (num_blocks < 0 || batch < 0 || out_capacity < 0 || bt_stride < 0) return IX_ERR_SHAPE;
    if (head_dim != kHeadDim || block_size != kBlockSize) return IX_ERR_UNSUPPORTED;
    if (batch == 0 || out_capacity == 0) return IX_OK;
    if (!cache || !block_table || !cu_seq_lens || !out_k || !out_scale) return IX_ERR_NULL;
    if (!aligned16(cache) || !aligned16(out_k) || (reinterpret_cast<uintptr_t>(out_scale) & 3))
        return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    gather_k_kernel<<<grid_for(out_capacity, 32), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        cache, num_blocks, block_table, bt_stride, cu_seq_lens, batch, out_k, out_scale,
        out_capacity, st);
    return launch_status();
}

extern "C" int dsmla_quant_write(const void* nope_bf16, const void* rope_bf16, int64_t n,
                                 const int64_t* slot_mapping, uint8_t* cache, int64_t num_blocks,
                                 int block_size, int64_t block_stride_bytes,
                                 int64_t entry_stride_bytes, ix_stream_t stream) {
    if (n < 0 || num_blocks < 0 || block_size <= 0 || block_stride_bytes <= 0 ||
        entry_stride_bytes < 656)
        return IX_ERR_SHAPE;
    if (n == 0) return IX_OK;
    if (!nope_bf16 || !rope_bf16 || !slot_mapping || !cache) return IX_ERR_NULL;
    if (!aligned16(nope_bf16) || !aligned16(rope_bf16) || !aligned16(cache) ||
        (block_stride_bytes & 15) || (entry_stride_bytes & 15) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
        return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    dsmla_write_kernel<<<grid_for(2 * n, 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(nope_bf16), static_cast<const uint4*>(rope_bf16), n, slot_mapping,
        cache, num_blocks, block_size, block_stride_bytes, entry_stride_bytes, st);
    return launch_status();
}

extern "C" int dsmla_norm_rope_write(const void* kv_bf16, const void* pe_bf16, const void* gamma_bf16,
                                     float eps, const int64_t* positions, const float* cos_sin,
                                     int64_t max_pos, const int64_t* slot_mapping, int64_t n,
                                     uint8_t* cache, int64_t num_blocks, int block_size,
                                     int64_t block_stride_bytes, int64_t entry_stride_bytes,
                                     ix_stream_t stream) {
    if (n < 0 || num_blocks < 0 || block_size <= 0 || block_stride_bytes <= 0 ||
        entry_stride_bytes < 656 || max_pos < 0)
        return IX_ERR_SHAPE;
    if (n == 0) return IX_OK;
    if (!kv_bf16 || !pe_bf16 || !gamma_bf16 || !positions || !cos_sin || !slot_mapping || !cache)
        return IX_ERR_NULL;
    if (!aligned16(kv_bf16) || !aligned16(gamma_bf16) || !aligned16(cache) ||
        (reinterpret_cast<uintptr_t>(pe_bf16) & 3) || (reinterpret_cast<uintptr_t>(cos_sin) & 3) ||
        (block_stride_bytes & 15) || (entry_stride_bytes & 15) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7) || (reinterpret_cast<uintptr_t>(positions) & 7))
        return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    dsmla_norm_rope_kernel<<<grid_for(n, 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(kv_bf16), static_cast<const uint32_t*>(pe_bf16),
        static_cast<const uint4*>(gamma_bf16), eps, positions, cos_sin, max_pos, slot_mapping, n, cache,
        num_blocks, block_size, block_stride_bytes, entry_stride_bytes, st);
    return launch_status();
}
