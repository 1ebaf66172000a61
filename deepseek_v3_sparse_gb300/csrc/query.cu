// query.cu -- the query side of the step.
//
//   dsmla_fused_q  the MQA query of the sparse MLA attention (vLLM PR #47090,
//                  prhub summary: fused_q's quantize_mqa flag selects an FP8 MQA
//                  query or the BF16 pair (ql_nope, q_pe)): q_pe is rotated as
//                  the cache's RoPE values are; with quantize_mqa the 576 values
//                  [ql_nope | rotated q_pe] are coded to fp8 with one
//                  amax / 448 scale per (token, head).
//   ix_quant_q     the indexer's fp8 query with its per-(token, head) amax / 448
//                  scale folded into the head weight (a positive scale commutes
//                  with the ReLU of the indexer score).
//
// Both are HBM-streaming: one warp per (token, head) for the MLA query (lane l
// holds ql_nope values 16l .. 16l + 15 and RoPE pair l), half a warp per
// (token, head) for the indexer query (lane holds 8 of the 128 values; four
// units' loads in flight per half-warp), 16-byte loads and stores, a shuffle
// max for amax.  Arithmetic: IEEE f32 products, sums and divisions (no fused
// multiply-add in the RoPE), bf16 and e4m3 conversions round to nearest even,
// e4m3 saturates.  The divisions by the scale are correctly rounded quotients
// obtained from one correctly rounded reciprocal per (token, head) and two
// FMAs per value (div_by_rcp).
#include <math.h>

#include "common.cuh"

namespace dsix {
namespace {

constexpr int kNope = 512;
constexpr int kRope = 64;
constexpr int kMqa = kNope + kRope;
constexpr int kQThreads = 256;
constexpr int kQUnroll = 4;  // indexer-query units per half-warp and iteration

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float warp_max(float v) {
    // non-negative values: their bit patterns order as the values do
    uint32_t u = __float_as_uint(v);
    u = __reduce_max_sync(0xffffffffu, u);
    return __uint_as_float(u);
}

// scale = max(amax / 448, FLT_MIN) with an IEEE division
__device__ __forceinline__ float scale_of(float amax) {
    const float s = __fdiv_rn(amax, 448.0f);
    return s >= 1.17549435e-38f ? s : 1.17549435e-38f;
}

// x / b rounded to nearest even, given y = RN(1/b).  Markstein's theorem for
// division with an FMA (P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990; see
// also Muller et al., Handbook of Floating-Point Arithmetic, the chapter on
// FMA-based division): q0 = RN(x y) is within one ulp of x / b, the residual
// x - b q0 is exact in one FMA, and RN(q0 + r y) is RN(x / b), as long as
// nothing underflows.  Used for b >= 2^-90 and |x / b| <= 448: then the
// residual is exact for every quotient of 2^-11 or more, and smaller quotients
// code to an e4m3 zero of the right sign whichever faithful value they get.
// The residual is formed as -(q0 b - x) so that x = -0 gives q0 = -0, a +0
// residual and the quotient -0 (x - q0 b would give +0 + -0 = +0).
__device__ __forceinline__ float div_by_rcp(float x, float b, float y) {
    const float q0 = __fmul_rn(x, y);
    const float rn = __fmaf_rn(q0, b, -x);  // -(x - b q0), exact
    return __fmaf_rn(-rn, y, q0);
}

// Divisions by one per-(token, head) scale, chosen once per (token, head): the
// reciprocal path above for scales of 2^-90 or more (every realistic scale),
// IEEE division below that.
struct RcpDiv {
    float sc, y;
    __device__ __forceinline__ float operator()(float x) const { return div_by_rcp(x, sc, y); }
};
struct IeeeDiv {
    float sc;
    __device__ __forceinline__ float operator()(float x) const { return __fdiv_rn(x, sc); }
};
constexpr float kRcpMinScale = 0x1p-90f;

struct FusedQArgs {
    const uint4* ql_nope;   // [T*H][64] uint4 (8 bf16 each)
    int heads_shift;        // log2(heads) when heads is a power of two, else -1
    const uint32_t* q_pe;   // [T*H][32] bf16 pairs
    const int64_t* positions;
    const float* cos_sin;
    int64_t max_pos;
    int64_t tokens;
    int heads;
    int quantize;
    uint32_t* out_pe;       // [T*H][32] bf16 pairs
    uint8_t* out_mqa;       // [T*H][576]
    float* out_scale;       // [T*H]
    int* status;
};

// e4m3 codes of a lane's 18 values: four words of the NoPE part, the RoPE pair
template <class Div>
__device__ __forceinline__ void mqa_codes(const float (&x)[18], const Div& dv, uint32_t (&code)[5]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
        code[i] = cvt_e4m3x2(dv(x[4 * i]), dv(x[4 * i + 1])) | (cvt_e4m3x2(dv(x[4 * i + 2]), dv(x[4 * i + 3])) << 16);
    code[4] = cvt_e4m3x2(dv(x[16]), dv(x[17]));
}

// e4m3 codes of a half-warp lane's 8 values (indexer query)
template <class Div>
__device__ __forceinline__ uint2 q_codes(const float (&x)[8], const Div& dv) {
    return make_uint2(cvt_e4m3x2(dv(x[0]), dv(x[1])) | (cvt_e4m3x2(dv(x[2]), dv(x[3])) << 16),
                      cvt_e4m3x2(dv(x[4]), dv(x[5])) | (cvt_e4m3x2(dv(x[6]), dv(x[7])) << 16));
}

__global__ void __launch_bounds__(kQThreads) fused_q_kernel(const FusedQArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t n = a.tokens * a.heads;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * (kQThreads / 32);
    for (int64_t th = static_cast<int64_t>(blockIdx.x) * (kQThreads / 32) + (threadIdx.x >> 5); th < n; th += nw) {
        const int64_t t = a.heads_shift >= 0 ? th >> a.heads_shift : th / a.heads;
        // loads first: the position, this lane's RoPE pair and NoPE values
        const int64_t p = __ldg(a.positions + t);
        const uint32_t pe = __ldg(a.q_pe + th * 32 + lane);
        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
        if (a.quantize) {
            v0 = __ldg(a.ql_nope + th * 64 + 2 * lane);
            v1 = __ldg(a.ql_nope + th * 64 + 2 * lane + 1);
        }
        if (p < 0 || p >= a.max_pos) {  // uniform over the warp
            if (lane == 0) flag(a.status, IX_DEV_BAD_POSITION);
            continue;
        }
        const float c = __ldg(a.cos_sin + p * 64 + lane), s = __ldg(a.cos_sin + p * 64 + 32 + lane);
        const float x0 = bf16_lo(pe), x1 = bf16_hi(pe);
        const float r1 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
        const float r2 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
        const uint32_t rot = bf16x2_rn(r1, r2);
        if (!a.quantize) {
            a.out_pe[th * 32 + lane] = rot;
            continue;
        }
        float x[18];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
        }
        x[16] = bf16_lo(rot);
        x[17] = bf16_hi(rot);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 18; ++i) amax = fmaxf(amax, fabsf(x[i]));
        const float sc = scale_of(warp_max(amax));
        uint32_t code[5];
        if (sc >= kRcpMinScale)  // uniform over the warp
            mqa_codes(x, RcpDiv{sc, __frcp_rn(sc)}, code);
        else
            mqa_codes(x, IeeeDiv{sc}, code);
        uint8_t* dst = a.out_mqa + th * kMqa;
        *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(code[0], code[1], code[2], code[3]);
        *reinterpret_cast<uint16_t*>(dst + kNope + 2 * lane) = static_cast<uint16_t>(code[4]);
        if (lane == 0) a.out_scale[th] = sc;
    }
}

// Indexer query: half a warp per (token, head) of 128 values, 8 per lane.
__global__ void __launch_bounds__(kQThreads) quant_q_kernel(const uint4* __restrict__ q, const float* __restrict__ w,
                                                            int64_t n, uint2* __restrict__ q_fp8,
                                                            float* __restrict__ w_out) {
    const int lane = threadIdx.x & 31, hl = lane & 15;
    const int64_t nh = static_cast<int64_t>(gridDim.x) * (kQThreads / 16);
    // Each half-warp takes kQUnroll (token, head) units per iteration, nh apart,
    // and issues all their loads before any arithmetic.  The loop test uses the
    // warp's first unit, so both halves of a warp walk it together (the shuffles
    // span the whole warp); a unit past the end computes on zeros and stores nothing.
    for (int64_t th0 = static_cast<int64_t>(blockIdx.x) * (kQThreads / 16) + (threadIdx.x >> 4);
         th0 - (lane >> 4) < n; th0 += kQUnroll * nh) {
        uint4 v[kQUnroll];
        float wt[kQUnroll];
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
            const int64_t th = th0 + u * nh;
            const bool live = th < n;
            v[u] = live ? __ldg(q + th * 16 + hl) : make_uint4(0u, 0u, 0u, 0u);
            wt[u] = live ? __ldg(w + th) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
            const int64_t th = th0 + u * nh;
            const float x[8] = {bf16_lo(v[u].x), bf16_hi(v[u].x), bf16_lo(v[u].y), bf16_hi(v[u].y),
                                bf16_lo(v[u].z), bf16_hi(v[u].z), bf16_lo(v[u].w), bf16_hi(v[u].w)};
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
            uint32_t m = __float_as_uint(amax);  // max over the 16 lanes of this half
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float sc = scale_of(__uint_as_float(m));
            if (th < n) {
                // the scale is uniform over the half-warp
                q_fp8[th * 16 + hl] =
                    sc >= kRcpMinScale ? q_codes(x, RcpDiv{sc, __frcp_rn(sc)}) : q_codes(x, IeeeDiv{sc});
                if (hl == 0) w_out[th] = __fmul_rn(wt[u], sc);
            }
        }
    }
}

int grid_for(int64_t units, int per_block) {
    const int sms = num_sms();
    if (sms <= 0) return -1;
    const int64_t need = (units + per_block - 1) / per_block;
    const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 blocks of 256 threads per SM
    return static_cast<int>(need < cap ? need : cap);
}

}  // namespace
}  // namespace dsix

using namespace dsix;

extern "C" int dsmla_fused_q(const void* ql_nope_bf16, const void* q_pe_bf16, const int64_t* positions,
                             const float* cos_sin, int64_t max_pos, int64_t tokens, int heads, int quantize_mqa,
                             void* out_pe_bf16, uint8_t* out_mqa_fp8, float* out_mqa_scale, ix_stream_t stream) {
    if (tokens < 0 || max_pos < 0) return IX_ERR_SHAPE;
    if (heads < 1) return IX_ERR_UNSUPPORTED;
    if (tokens == 0) return IX_OK;
    if (tokens * heads >= (1ll << 40)) return IX_ERR_UNSUPPORTED;
    if (!q_pe_bf16 || !positions || (max_pos > 0 && !cos_sin)) return IX_ERR_NULL;
    if (quantize_mqa ? (!ql_nope_bf16 || !out_mqa_fp8 || !out_mqa_scale) : !out_pe_bf16) return IX_ERR_NULL;
    auto al = [](const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
    if (!al(q_pe_bf16, 4) || !al(positions, 8) || !al(cos_sin, 4)) return IX_ERR_ALIGN;
    if (quantize_mqa ? (!al(ql_nope_bf16, 16) || !al(out_mqa_fp8, 16) || !al(out_mqa_scale, 4))
                     : !al(out_pe_bf16, 4))
        return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    FusedQArgs a{};
    a.ql_nope = static_cast<const uint4*>(ql_nope_bf16);
    a.q_pe = static_cast<const uint32_t*>(q_pe_bf16);
    a.positions = positions;
    a.cos_sin = cos_sin;
    a.max_pos = max_pos;
    a.tokens = tokens;
    a.heads = heads;
    a.heads_shift = (heads & (heads - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(heads)) : -1;
    a.quantize = quantize_mqa ? 1 : 0;
    a.out_pe = static_cast<uint32_t*>(out_pe_bf16);
    a.out_mqa = out_mqa_fp8;
    a.out_scale = out_mqa_scale;
    a.status = st;
    const int grid = grid_for(tokens * heads, kQThreads / 32);
    if (grid <= 0) return IX_ERR_CUDA;
    fused_q_kernel<<<grid, kQThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return launch_status();
}

extern "C" int ix_quant_q(const void* q_bf16, const float* w, int64_t tokens, int heads, int head_dim,
                          uint8_t* q_fp8, float* w_out, ix_stream_t stream) {
    if (tokens < 0) return IX_ERR_SHAPE;
    if (heads < 1 || head_dim != 128) return IX_ERR_UNSUPPORTED;
    if (tokens == 0) return IX_OK;
    if (tokens * heads >= (1ll << 40)) return IX_ERR_UNSUPPORTED;
    if (!q_bf16 || !w || !q_fp8 || !w_out) return IX_ERR_NULL;
    if (!aligned16(q_bf16) || (reinterpret_cast<uintptr_t>(q_fp8) & 7u) || (reinterpret_cast<uintptr_t>(w) & 3u) ||
        (reinterpret_cast<uintptr_t>(w_out) & 3u))
        return IX_ERR_ALIGN;
    const int64_t n = tokens * heads;
    const int grid = grid_for(n, kQThreads / 16);
    if (grid <= 0) return IX_ERR_CUDA;
    quant_q_kernel<<<grid, kQThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(q_bf16), w, n, reinterpret_cast<uint2*>(q_fp8), w_out);
    return launch_status();
}
