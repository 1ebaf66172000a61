// sparse_mla.cu -- sparse MLA decode attention over the fp8_ds_mla cache.
//
// The consumer of the global top-k indices: for query token t and head h,
// softmax attention of the bf16 query (ql_nope [512], q_pe [64]) over the
// 656-byte cache entries named by row t of the index buffer (vLLM PR #47090,
// prhub summary: the fp8_ds_mla layout and the bf16 query pair; ROCm/ATOM PR
// #1094, Technical Details: per-query global paged-KV indices).  Entry of slot g:
//   k[i] = e4m3(code[i]) * scale[i / 128]  (i < 512),  k[512 + i] = rope[i],
//   v = k[0, 512);  z_j = sm_scale * (q . k_j);
//   out = sum_j softmax(z)_j v_j,  lse = log sum_j exp(z_j)  (natural log).
// A negative index names no key; a token with no key gets out = 0, lse = -inf.
//
// GPU layout: one CTA per (token, split of 256 indices), 448 threads, one CTA
// per SM (512 TMEM columns, ~195 KB of shared memory).
//   warp 0      MMA issuer (one lane elected once) and TMEM owner
//   warp 1      TMA producer of the query chunks (bf16, 128-byte swizzle)
//   warps 2-9   dequantisers: fp8 x tile scale -> bf16 operand tiles written
//               into shared memory in the 128-byte-swizzled K-major layout
//   warps 10-13 softmax and epilogue, one thread per head (= TMEM lane)
// Phase 1  S[128 heads x 256 keys] = Q K^T (tcgen05 kind::f16, M 128, N 256)
//          into TMEM columns [0, 256), over nine 64-dim chunks (the RoPE
//          chunk, then eight NoPE chunks): query chunks in a ring of four
//          (TMA), bf16 key chunks in two stages, the gathered codes ahead
//          by cp.async in a ring of four, all in the space of the V^T tiles
//          and P (both free until S is complete).
// Phase 2  the softmax threads read their row of S twice (max, then
//          exponentials by the hardware approximation), write P in bf16 as the
//          A operand of the next product and keep the row sums.
// Phase 3  O[128 x 512] = P V into TMEM columns [0, 512) (S has been read by
//          then): four chunks of 64 keys, V^T tiles [512 dims x 64 keys]
//          written by the dequantisers, two N = 256 halves per K step.
// Epilogue O / sum (32 x 32 tiles, 128-byte swizzled, stored by TMA) and the
//          split's lse go to the caller's workspace; a second kernel, launched
//          as this one's programmatic dependent, merges the splits of each
//          (token, head) into bf16 output.
// Every wait is bounded (IX_DEV_TIMEOUT, then all roles leave; in-flight
// copies and MMAs are drained before the CTA frees its TMEM and exits).
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace dsix {
namespace {

constexpr int kH = 128;        // heads = MMA M
constexpr int kNope = 512;
constexpr int kEntry = 656;    // bytes of one entry: codes, 4 scales, RoPE
constexpr int kSplit = 256;    // indices per CTA = N of the first product
constexpr int kChunks = 9;     // 64-dim chunks of the 576-dim dot product
constexpr int kKeyChunks = kSplit / 64;
constexpr int kMaxTopk = 65536;
constexpr int kThreads = 448;
constexpr int kMmaWarp = 0, kTmaWarp = 1, kDeqWarp0 = 2, kDeqWarps = 8, kSmWarp0 = 10;
constexpr int kDeqThreads = kDeqWarps * 32;
static_assert(kSmWarp0 == kDeqWarp0 + kDeqWarps && (kSmWarp0 + 4) * 32 == kThreads,
              "four softmax warps after the dequantisers cover the 128 TMEM lanes");
static_assert(kDeqThreads == kSplit, "one dequantiser thread per key of a split");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s

// shared memory map (offsets from a 1024-byte-aligned base)
constexpr int kQBytes = kH * 128;                 // one 64-dim query chunk (16 KB)
constexpr int kKBytes = kSplit * 128;             // one 64-dim key chunk (32 KB)
// Phase 1 uses the V^T region and the P tiles (both free until S is complete):
constexpr int kQStages = 4;                       // query chunks in flight (TMA)
constexpr int kP1Stages = 2;                      // bf16 key chunk stages (written by the dequantisers)
constexpr int kRing = 4;                          // chunks of gathered codes in flight (cp.async)
constexpr int kKStageOff = kQStages * kQBytes;    // after the query ring
constexpr int kRingOff = kKStageOff + kP1Stages * kKBytes;  // [kRing][256 keys x 64 codes]
constexpr int kVtBytes = kNope * 128;             // V^T tile: 512 rows x 64 keys (64 KB)
constexpr int kRegion = 2 * kVtBytes;             // both V^T stages (phase 1: query ring, key stages)
constexpr int kPOff = kRegion;                    // P: 4 tiles of 128 rows x 64 keys
constexpr int kPAtom = kH * 128;
constexpr int kOffOff = kPOff + kKeyChunks * kPAtom;  // int64 entry offset per key (-1: none)
constexpr int kMaskOff = kOffOff + kSplit * 8;        // validity bits of the 256 keys
constexpr int kBarOff = kMaskOff + 64;
constexpr int kNumBars = 2 * kQStages + 2 * kP1Stages + 8;
constexpr int kMiscOff = kBarOff + kNumBars * 8;      // tmem base, abort flag, never-raised flag
constexpr int kSmemUsed = kMiscOff + 64;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kRingOff + kRing * kSplit * 64 <= kOffOff, "phase-1 stages and code ring fit the V^T region and P");
static_assert(kSmemAlloc <= 232448, "shared memory per CTA");

struct SmlaArgs {
    const uint8_t* cache;
    int64_t num_blocks;
    int64_t block_stride;
    int64_t entry_stride;
    const int32_t* indices;
    int64_t tokens;
    int block_size;
    int topk;
    int splits;
    float scale_log2;  // sm_scale * log2(e)
    float* ws_o;       // [tokens * splits * 128, 512]: O / row sum of each split
    float* ws_lse;     // [tokens * splits * 128]: natural-log sum of exponentials
    int* status;
};

// ---------------------------------------------------------------------------
// small device helpers of this file
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// Instruction descriptor, kind::f16: A = B = BF16, D = F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                // D format: F32
           | (1u << 7) | (1u << 10)                 // A, B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// bf16x2 of (lo, hi), round to nearest even; lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 2^x by the hardware's approximate exponential; results below 2^-126 are
// flushed to zero.
__device__ __forceinline__ float ex2_ftz(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Two e4m3 codes (low byte = first) -> their exact values as f32.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float& lo, float& hi) {
    uint32_t h2;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h2) : "r"(two));
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
}

// Four codes (bytes of w, first in the low byte) times one scale -> 4 bf16.
__device__ __forceinline__ uint2 deq4(uint32_t w, float sc) {
    float a, b, c, d;
    e4m3x2_to_f32(w & 0xFFFFu, a, b);
    e4m3x2_to_f32(w >> 16, c, d);
    return make_uint2(pack_bf16(a * sc, b * sc), pack_bf16(c * sc, d * sc));
}

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag (drains in-flight work on the way out);
// `never` points at a shared-memory word that stays 0.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, volatile int* never, int* status) {
    mbar_wait(bar, parity, never, status, kDrainLimitNs);
}

// ---------------------------------------------------------------------------
// main kernel: one CTA per (token, split)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    smla_decode_kernel(const __grid_constant__ CUtensorMap tmQn, const __grid_constant__ CUtensorMap tmQp,
                       const __grid_constant__ CUtensorMap tmO, const SmlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int64_t* koff = reinterpret_cast<int64_t*>(sm + kOffOff);
    uint32_t* vmask = reinterpret_cast<uint32_t*>(sm + kMaskOff);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBarOff);
    uint64_t* qfull = bars;                   // [kQStages] query chunk landed
    uint64_t* qempty = qfull + kQStages;      // [kQStages] the MMAs reading a query chunk are done
    uint64_t* full1 = qempty + kQStages;      // [kP1Stages] key chunk written
    uint64_t* empty1 = full1 + kP1Stages;     // [kP1Stages] the MMAs of a key stage are done
    uint64_t* s_full = empty1 + kP1Stages;    // all of S is in TMEM (phase-1 MMAs done)
    uint64_t* p_full = s_full + 1;            // P written, S read (128 softmax threads)
    uint64_t* full3 = s_full + 2;             // [2] V^T chunk written
    uint64_t* empty3 = s_full + 4;            // [2] the MMAs of a V^T stage are done
    uint64_t* o_full = s_full + 6;            // O complete in TMEM
    uint64_t* mma_done = s_full + 7;
    int* misc = reinterpret_cast<int*>(sm + kMiscOff);
    volatile int* abort_flag = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x / a.splits;
    const int split = static_cast<int>(blockIdx.x % a.splits);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(qfull + i, 1);
            mbar_init(qempty + i, 1);
        }
        for (int i = 0; i < kP1Stages; ++i) {
            mbar_init(full1 + i, kDeqThreads);
            mbar_init(empty1 + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(full3 + i, kDeqThreads);
            mbar_init(empty3 + i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, kH);
        mbar_init(o_full, 1);
        mbar_init(mma_done, 1);
        fence_barrier_init();
        misc[1] = 0;
        misc[2] = 0;  // never raised: the abort flag seen by drain waits
    }
    if (warp == kTmaWarp && lane == 0) {
        prefetch_tmap(&tmQn);
        prefetch_tmap(&tmQp);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), kTmemCols);
        tmem_relinquish();
    }
    // this split's indices -> entry byte offsets (-1: no key); each entry is
    // pulled into L2 now, so the dequantisers' chunk loads hit L2
    if (threadIdx.x < kSplit) {
        const int j = split * kSplit + threadIdx.x;
        int64_t off = -1;
        if (j < a.topk) {
            const int64_t g = __ldg(a.indices + t * a.topk + j);
            if (g >= 0) {
                const int64_t blk = g / a.block_size;
                if (blk < a.num_blocks) {
                    off = blk * a.block_stride + (g - blk * a.block_size) * a.entry_stride;
                    prefetch_l2(a.cache + off, kEntry);
                } else {
                    flag(a.status, IX_DEV_BAD_SLOT);
                }
            }
        }
        koff[threadIdx.x] = off;
        const uint32_t bal = __ballot_sync(0xffffffffu, off >= 0);
        if (lane == 0) vmask[threadIdx.x >> 5] = bal;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);
    pdl_trigger();  // the merge kernel may be scheduled now; it waits for this grid's end

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ query chunks
        const bool leader = elect_one();
        int c = 0;
        for (; c < kChunks; ++c) {
            const int stage = c % kQStages, use = c / kQStages;
            if (use > 0 && !wait_warp(qempty + stage, (use - 1) & 1, abort_flag, a.status)) break;
            if (leader) {
                uint8_t* qdst = sm + stage * kQBytes;
                mbar_arrive_expect_tx(qfull + stage, kQBytes);
                if (c == 0)  // chunk 0: the RoPE part; chunks 1-8: NoPE dims 64 (c - 1) ..
                    tma_load_2d(qdst, &tmQp, qfull + stage, 0, static_cast<int>(t * kH));
                else
                    tma_load_2d(qdst, &tmQn, qfull + stage, (c - 1) * 64, static_cast<int>(t * kH));
            }
            __syncwarp();
        }
        // drain: the last copies issued must land before the CTA exits
        if (leader)
            for (int i = c > kQStages ? c - kQStages : 0; i < c; ++i)
                drain_wait(qfull + i % kQStages, (i / kQStages) & 1, misc + 2, a.status);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        constexpr uint32_t kId = idesc_bf16_f32(kH, 256);
        bool ok = true, issued = false;
        for (int c = 0; c < kChunks; ++c) {
            const int stage = c % kP1Stages, qs = c % kQStages;
            if (!wait_warp(qfull + qs, (c / kQStages) & 1, abort_flag, a.status) ||
                !wait_warp(full1 + stage, (c / kP1Stages) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t qa = smem_u32(sm + qs * kQBytes), kb = smem_u32(sm + kKStageOff + stage * kKBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem_base, sdesc_k_sw128(qa + 32 * kk), sdesc_k_sw128(kb + 32 * kk), kId,
                             (c | kk) != 0);
                mma_commit(qempty + qs);
                mma_commit(empty1 + stage);
            }
            issued = true;
            __syncwarp();
        }
        if (ok) {
            if (leader) mma_commit(s_full);
            __syncwarp();
            ok = wait_warp(p_full, 0, abort_flag, a.status);
        }
        for (int kc = 0; kc < kKeyChunks && ok; ++kc) {
            const int stage = kc & 1;
            if (!wait_warp(full3 + stage, (kc >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint32_t pa = smem_u32(sm + kPOff + kc * kPAtom), vb = smem_u32(sm + stage * kVtBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_k_sw128(pa + 32 * kk);
                    mma_bf16(tmem_base, ad, sdesc_k_sw128(vb + 32 * kk), kId, (kc | kk) != 0);
                    mma_bf16(tmem_base + 256, ad, sdesc_k_sw128(vb + kVtBytes / 2 + 32 * kk), kId, (kc | kk) != 0);
                }
                mma_commit(empty3 + stage);
            }
            __syncwarp();
        }
        if (ok) {
            if (leader) mma_commit(o_full);
            __syncwarp();
        }
        if (issued) {
            if (leader) {
                mma_commit(mma_done);
                drain_wait(mma_done, 0, misc + 2, a.status);
            }
            __syncwarp();
        }
    } else if (warp < kDeqWarp0 + kDeqWarps) {
        // ------------------------------------------------------------ dequantisers
        const int i = threadIdx.x - kDeqWarp0 * 32;
        bool ok = true;
        {
            // phase 1: four threads per key -- thread i covers keys 64 p + i / 4
            // (p = 0..3) and, of each 64-dim chunk, the 16 dims 16 (i % 4) ..,
            // i.e. two 16-byte pieces of the key's 128-byte operand row.  The
            // codes travel by cp.async (16 bytes per key and chunk, no register
            // round trip) into a ring of kRing chunks, so up to kRing chunks of
            // gathered codes are in flight per CTA; a thread converts only the
            // bytes it copied itself.  Chunk 0 is the RoPE part, copied as stored
            // straight into its place in stage 0's tile; chunks 1-8 are the NoPE
            // codes times their tile scale.  A key without an entry gives zeros.
            const int qtr = i & 3, kb = i >> 2;
            const uint8_t* ent[4];
            bool valid[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int64_t off = koff[p * 64 + kb];
                valid[p] = off >= 0;
                ent[p] = a.cache + (valid[p] ? off : 0);
            }
            uint4* ring = reinterpret_cast<uint4*>(sm + kRingOff);  // [kRing][4 keys][256 threads]
            {
                uint8_t* kt = sm + kKStageOff;  // key stage 0, first use
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int row = p * 64 + kb;
                    uint8_t* d0 = kt + row * 128 + (((2 * qtr) ^ (row & 7)) << 4);
                    uint8_t* d1 = kt + row * 128 + (((2 * qtr + 1) ^ (row & 7)) << 4);
                    if (valid[p]) {
                        const uint8_t* rope = ent[p] + kNope + 16 + qtr * 32;
                        cp_async16(d0, rope);
                        cp_async16(d1, rope + 16);
                    } else {
                        *reinterpret_cast<uint4*>(d0) = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4*>(d1) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                cp_async_commit();
            }
            auto fetch = [&](int n) {  // NoPE chunk n's codes -> ring slot n % kRing (one group, maybe empty)
                if (n < 8) {
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        if (valid[p]) cp_async16(ring + ((n % kRing) * 4 + p) * 256 + i, ent[p] + n * 64 + qtr * 16);
                }
                cp_async_commit();
            };
#pragma unroll
            for (int n = 0; n < kRing; ++n) fetch(n);
            float4 sc[4];  // the four tile scales of each key
#pragma unroll
            for (int p = 0; p < 4; ++p)
                sc[p] = valid[p] ? __ldg(reinterpret_cast<const float4*>(ent[p] + kNope)) : make_float4(0.f, 0.f, 0.f, 0.f);
            uint4 o[8];
            auto put_rows = [&](int stage) {
                uint8_t* kt = sm + kKStageOff + stage * kKBytes;
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int row = p * 64 + kb;
                    uint8_t* krow = kt + row * 128;
                    *reinterpret_cast<uint4*>(krow + (((2 * qtr) ^ (row & 7)) << 4)) = o[2 * p];
                    *reinterpret_cast<uint4*>(krow + (((2 * qtr + 1) ^ (row & 7)) << 4)) = o[2 * p + 1];
                }
                fence_proxy_async();
                mbar_arrive(full1 + stage);
            };
            // chunk 0: its copies are the oldest group
            cp_async_wait<kRing>();
            fence_proxy_async();
            mbar_arrive(full1 + 0);
#pragma unroll
            for (int n = 0; n < 8; ++n) {  // unrolled: slots, scales and stages are constants
                if (!ok) break;
                const int c = n + 1, stage = c % kP1Stages, use = c / kP1Stages;
                cp_async_wait<kRing - 1>();  // this thread's copies of chunk n have landed
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const float s4 = (n >> 1) == 0 ? sc[p].x : (n >> 1) == 1 ? sc[p].y : (n >> 1) == 2 ? sc[p].z : sc[p].w;
                    uint4 r = make_uint4(0u, 0u, 0u, 0u);
                    if (valid[p]) r = ring[((n % kRing) * 4 + p) * 256 + i];
                    const uint2 a0 = deq4(r.x, s4), a1 = deq4(r.y, s4), a2 = deq4(r.z, s4), a3 = deq4(r.w, s4);
                    o[2 * p] = make_uint4(a0.x, a0.y, a1.x, a1.y);
                    o[2 * p + 1] = make_uint4(a2.x, a2.y, a3.x, a3.y);
                }
                // the slot's codes are in registers (the dependency below orders the
                // shared loads before the refill's copies)
                asm volatile("" ::"r"(o[0].x), "r"(o[2].x), "r"(o[4].x), "r"(o[6].x) : "memory");
                fetch(n + kRing);
                if (use > 0 && !wait_warp(empty1 + stage, (use - 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                put_rows(stage);
            }
            cp_async_wait_all();  // nothing of phase 1 lands in shared memory after this point
        }
        // phase 3: V^T tiles; thread i covers 8 keys (g) x 16 dims (e) of a
        // 64-key chunk.  Chunk 0's codes are loaded before the wait for S, and
        // each later chunk's right after the previous one is stored (one
        // register set: a second one spills at this kernel's register budget).
        // The shared region is reused, so nothing is written before every
        // phase-1 MMA has read it (s_full).
        const int g = i & 7, e = i >> 3;
        uint32_t wa[8][4];
        float sc[8];  // tile scales of the 8 keys, loaded with their codes
        auto load_v = [&](int kc, uint32_t(&w)[8][4]) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int64_t ko = koff[kc * 64 + g * 8 + kk];
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                sc[kk] = 0.0f;
                if (ko >= 0) {
                    v = __ldg(reinterpret_cast<const uint4*>(a.cache + ko + e * 16));
                    sc[kk] = __ldg(reinterpret_cast<const float*>(a.cache + ko + kNope) + (e >> 3));
                }
                w[kk][0] = v.x;
                w[kk][1] = v.y;
                w[kk][2] = v.z;
                w[kk][3] = v.w;
            }
        };
        auto put_v = [&](int kc, const uint32_t(&w)[8][4]) -> bool {
            const int stage = kc & 1, use = kc >> 1;
            if (use > 0 && !wait_warp(empty3 + stage, (use - 1) & 1, abort_flag, a.status)) return false;
            uint8_t* vt = sm + stage * kVtBytes;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int d = e * 16 + r;
                const uint32_t sel = static_cast<uint32_t>((r & 3) | ((4 + (r & 3)) << 4));
                uint32_t ow[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    float lo, hi;
                    e4m3x2_to_f32(__byte_perm(w[2 * p][r >> 2], w[2 * p + 1][r >> 2], sel), lo, hi);
                    ow[p] = pack_bf16(lo * sc[2 * p], hi * sc[2 * p + 1]);
                }
                *reinterpret_cast<uint4*>(vt + d * 128 + ((g ^ (d & 7)) << 4)) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
            fence_proxy_async();
            mbar_arrive(full3 + stage);
            return true;
        };
        load_v(0, wa);  // registers only: may run before the region is free
        if (ok) ok = wait_warp(s_full, 0, abort_flag, a.status);
        for (int kc = 0; kc < kKeyChunks && ok; ++kc) {
            if (kc > 0) load_v(kc, wa);
            ok = put_v(kc, wa);
        }
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        const int q4 = warp & 3;
        const int h = q4 * 32 + lane;
        const uint32_t trow = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
        float m = -INFINITY, mc = 0.0f, l_exact = 0.0f, l_used = 0.0f;
        bool ok = wait_warp(s_full, 0, abort_flag, a.status);
        if (ok) {
            tc_fence_after();
            // pass 1: row max over the keys with an entry, two TMEM chunks per wait
            for (int cc = 0; cc < kSplit / 32; cc += 2) {
                uint32_t r0[32], r1[32];
                tmem_ld32(trow + cc * 32, r0);
                tmem_ld32(trow + (cc + 1) * 32, r1);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
                const uint32_t v0 = vmask[cc], v1 = vmask[cc + 1];
                if ((v0 & v1) == 0xffffffffu) {
                    float m0 = m, m1 = -INFINITY;
#pragma unroll
                    for (int k = 0; k < 32; k += 2) {
                        m0 = fmaxf(m0, fmaxf(__uint_as_float(r0[k]), __uint_as_float(r0[k + 1])));
                        m1 = fmaxf(m1, fmaxf(__uint_as_float(r1[k]), __uint_as_float(r1[k + 1])));
                    }
                    m = fmaxf(m0, m1);
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        if ((v0 >> k) & 1u) m = fmaxf(m, __uint_as_float(r0[k]));
                        if ((v1 >> k) & 1u) m = fmaxf(m, __uint_as_float(r1[k]));
                    }
                }
            }
            // sm_scale > 0, so the max of the scaled scores is the scaled max
            mc = m == -INFINITY ? 0.0f : m * a.scale_log2;
            uint8_t* prow = sm + kPOff + h * 128;
            // pass 2: P = 2^(s scale_log2 - mc) in bf16 (exponentials below 2^-126
            // flush to zero: far below the row's largest term, which is 1), the
            // row sums of the exact and of the rounded values in two partial sums each
            float le[2] = {0.0f, 0.0f}, lu[2] = {0.0f, 0.0f};
            for (int cc = 0; cc < kSplit / 32; ++cc) {
                uint32_t r[32];
                tmem_ld32(trow + cc * 32, r);
                tmem_wait_ld(r);
                const uint32_t vm = vmask[cc];
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {
                    float p0 = ex2_ftz(fmaf(__uint_as_float(r[k]), a.scale_log2, -mc));
                    float p1 = ex2_ftz(fmaf(__uint_as_float(r[k + 1]), a.scale_log2, -mc));
                    if (vm != 0xffffffffu) {
                        p0 = ((vm >> k) & 1u) ? p0 : 0.0f;
                        p1 = ((vm >> (k + 1)) & 1u) ? p1 : 0.0f;
                    }
                    le[(k >> 1) & 1] += p0 + p1;
                    const uint32_t b = pack_bf16(p0, p1);
                    lu[(k >> 1) & 1] += __uint_as_float(b << 16) + __uint_as_float(b & 0xFFFF0000u);
                    pk[k >> 1] = b;
                }
                uint8_t* atom = prow + (cc >> 1) * kPAtom;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = (cc & 1) * 4 + q;
                    *reinterpret_cast<uint4*>(atom + ((j ^ (h & 7)) << 4)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            l_exact = le[0] + le[1];
            l_used = lu[0] + lu[1];
            tc_fence_before();
            fence_proxy_async();
            mbar_arrive(p_full);
            ok = wait_warp(o_full, 0, abort_flag, a.status);
        }
        if (ok) {
            tc_fence_after();
            const float inv = l_used > 0.0f ? 1.0f / l_used : 0.0f;
            const int64_t prow_idx = (t * a.splits + split) * kH + h;
            // Rows leave by TMA (the V^T region is free once O is complete): a warp
            // writes 32 heads x 32 columns of O / sum into a 4 KB tile in the
            // 128-byte-swizzled layout of the split-output map, and one lane
            // stores it as a box; four tiles per warp rotate, a pair per step.
            uint8_t* tiles = sm + q4 * (4 * 4096);
            const int row0 = static_cast<int>(prow_idx - lane);  // the warp's first head row
            for (int cc = 0; cc < kNope / 32; cc += 2) {
                uint32_t r0[32], r1[32];
                tmem_ld32(trow + cc * 32, r0);
                tmem_ld32(trow + (cc + 1) * 32, r1);
                tmem_wait_ld(r0);
                tmem_wait_ld(r1);
                uint8_t* t0 = tiles + ((cc >> 1) & 1) * 8192;
                if (cc >= 4) {  // the pair stored from these tiles two steps ago has been read
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int pos = ((j ^ (lane & 7)) << 4);
                    *reinterpret_cast<float4*>(t0 + lane * 128 + pos) =
                        make_float4(__uint_as_float(r0[4 * j]) * inv, __uint_as_float(r0[4 * j + 1]) * inv,
                                    __uint_as_float(r0[4 * j + 2]) * inv, __uint_as_float(r0[4 * j + 3]) * inv);
                    *reinterpret_cast<float4*>(t0 + 4096 + lane * 128 + pos) =
                        make_float4(__uint_as_float(r1[4 * j]) * inv, __uint_as_float(r1[4 * j + 1]) * inv,
                                    __uint_as_float(r1[4 * j + 2]) * inv, __uint_as_float(r1[4 * j + 3]) * inv);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmO, t0, cc * 32, row0);
                    tma_store_2d(&tmO, t0 + 4096, (cc + 1) * 32, row0);
                    bulk_commit();
                }
            }
            if (lane == 0) bulk_wait_all();  // the splits are written before the CTA ends
            __syncwarp();
            a.ws_lse[prow_idx] = m == -INFINITY ? -INFINITY : (mc + log2f(l_exact)) * 0.69314718055994531f;
        } else {
            // a wait gave up: this split's output was not written, so its lse is
            // set to -inf and the merge gives it weight 0 (IX_DEV_TIMEOUT is set)
            a.ws_lse[(t * a.splits + split) * kH + h] = -INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// split merge: one warp per (token, head); lane l owns dims 4 (l + 32 q) .. +3
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
    smla_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_lse, int64_t rows,
                        int splits, uint16_t* __restrict__ out, float* __restrict__ lse) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_wait();  // launched as the main kernel's dependent: its split outputs are complete here
    if (row >= rows) return;
    const int64_t t = row / kH;
    const int h = static_cast<int>(row % kH);
    float M = -INFINITY;
    for (int s = lane; s < splits; s += 32) M = fmaxf(M, __ldg(ws_lse + (t * splits + s) * kH + h));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float4 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.0f;
    if (M != -INFINITY) {
        // four splits per round, all their loads in flight before the sums; a
        // split without keys has weight 0 and an all-zero output
        for (int s0 = 0; s0 < splits; s0 += 4) {
            float w[4];
            float4 v[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = s0 + j;
                w[j] = 0.0f;
#pragma unroll
                for (int q = 0; q < 4; ++q) v[j][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s < splits) {
                    const int64_t pr = (t * splits + s) * kH + h;
                    const float ls = __ldg(ws_lse + pr);
                    w[j] = ls == -INFINITY ? 0.0f : expf(ls - M);
                    const float4* src = reinterpret_cast<const float4*>(ws_o + pr * kNope);
#pragma unroll
                    for (int q = 0; q < 4; ++q) v[j][q] = __ldg(src + lane + 32 * q);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (s0 + j >= splits || w[j] == 0.0f) continue;
                L += w[j];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[q].x = fmaf(w[j], v[j][q].x, acc[q].x);
                    acc[q].y = fmaf(w[j], v[j][q].y, acc[q].y);
                    acc[q].z = fmaf(w[j], v[j][q].z, acc[q].z);
                    acc[q].w = fmaf(w[j], v[j][q].w, acc[q].w);
                }
            }
        }
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    uint2* dst = reinterpret_cast<uint2*>(out + row * kNope);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        dst[lane + 32 * q] = make_uint2(pack_bf16(acc[q].x * inv, acc[q].y * inv), pack_bf16(acc[q].z * inv, acc[q].w * inv));
    if (lane == 0) lse[row] = M == -INFINITY ? -INFINITY : M + logf(L);
}

// File-scope scratch of dsmla_sparse_decode_noalloc: room for the split
// outputs of kStaticSplits (token, split) pairs -- a decode batch of 16 tokens
// at top-2048 -- 33.6 MB of device memory, placed when this module loads.
constexpr int64_t kStaticSplits = 128;
static __device__ __align__(256) float g_smla_scratch[kStaticSplits * kH * (kNope + 1)];

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 map over rows of `cols` values (row pitch `cols` * 2 bytes), box of
// 64 values x 128 rows, 128-byte swizzle: one query chunk lands in the MMA's
// K-major layout.
bool make_query_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[2] = {cols, rows};
    cuuint64_t s[1] = {cols * 2};
    cuuint32_t b[2] = {64, static_cast<cuuint32_t>(kH)};
    cuuint32_t e[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), d, s, b, e,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split outputs [rows, 512] f32 as boxes of 32 rows x 32 columns (128-byte rows).
bool make_split_map(CUtensorMap* m, float* base, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[2] = {static_cast<cuuint64_t>(kNope), rows};
    cuuint64_t s[1] = {static_cast<cuuint64_t>(kNope) * 4};
    cuuint32_t b[2] = {32, 32};
    cuuint32_t e[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int smem_setup() {  // the dynamic shared memory limit, once per device
    static std::mutex mu;
    static std::vector<char> ready;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(ready.size())) ready.resize(dev + 1, 0);
    if (!ready[dev]) {
        if (cudaFuncSetAttribute(smla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) !=
            cudaSuccess)
            return IX_ERR_CUDA;
        ready[dev] = 1;
    }
    return IX_OK;
}

}  // namespace
}  // namespace dsix

using namespace dsix;

extern "C" size_t dsmla_sparse_decode_workspace_size(int64_t tokens, int heads, int topk) {
    if (tokens <= 0 || heads <= 0 || topk <= 0) return 0;
    const int64_t splits = (static_cast<int64_t>(topk) + kSplit - 1) / kSplit;
    return static_cast<size_t>(tokens * splits * heads) * (kNope + 1) * sizeof(float);
}

namespace dsix {
namespace {
// The argument checks both sparse decode entry points run first, in this
// order; `empty` is set when tokens == 0 (nothing to do, IX_OK).
int smla_check(const void* q_nope_bf16, const void* q_pe_bf16, const uint8_t* cache, int64_t num_blocks,
               int block_size, int64_t block_stride_bytes, int64_t entry_stride_bytes, const int32_t* indices,
               int64_t tokens, int heads, int topk, float sm_scale, const void* out_bf16, const float* lse,
               bool* empty) {
    *empty = false;
    if (tokens < 0 || num_blocks < 0 || block_stride_bytes < 0 || entry_stride_bytes < 0 || topk < 0)
        return IX_ERR_SHAPE;
    if (heads != kH || block_size < 1 || topk < 1 || topk > kMaxTopk) return IX_ERR_UNSUPPORTED;
    if (!(sm_scale > 0.0f) || !isfinite(sm_scale)) return IX_ERR_UNSUPPORTED;
    if (tokens == 0) {
        *empty = true;
        return IX_OK;
    }
    if (!q_nope_bf16 || !q_pe_bf16 || !indices || !out_bf16 || !lse || (num_blocks > 0 && !cache)) return IX_ERR_NULL;
    if (entry_stride_bytes < kEntry || block_stride_bytes < static_cast<int64_t>(block_size) * entry_stride_bytes)
        return IX_ERR_SHAPE;
    if (!aligned16(q_nope_bf16) || !aligned16(q_pe_bf16) || !aligned16(cache) || !aligned16(out_bf16) ||
        (block_stride_bytes & 15) || (entry_stride_bytes & 15) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(indices) & 3u))
        return IX_ERR_ALIGN;
    const int64_t splits = (static_cast<int64_t>(topk) + kSplit - 1) / kSplit;
    if (tokens * kH > INT32_MAX || tokens * splits > INT32_MAX) return IX_ERR_UNSUPPORTED;
    return IX_OK;
}
}  // namespace
}  // namespace dsix

extern "C" int dsmla_sparse_decode(const void* q_nope_bf16, const void* q_pe_bf16, const uint8_t* cache,
                                   int64_t num_blocks, int block_size, int64_t block_stride_bytes,
                                   int64_t entry_stride_bytes, const int32_t* indices, int64_t tokens, int heads,
                                   int topk, float sm_scale, void* out_bf16, float* lse, void* workspace,
                                   size_t workspace_bytes, ix_stream_t stream) {
    bool empty = false;
    const int chk = smla_check(q_nope_bf16, q_pe_bf16, cache, num_blocks, block_size, block_stride_bytes,
                               entry_stride_bytes, indices, tokens, heads, topk, sm_scale, out_bf16, lse, &empty);
    if (chk != IX_OK || empty) return chk;
    const int splits = (topk + kSplit - 1) / kSplit;
    const int64_t prow = tokens * splits * kH;
    const size_t need = dsmla_sparse_decode_workspace_size(tokens, heads, topk);
    if (!workspace || workspace_bytes < need) return IX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return IX_ERR_ALIGN;
    int* status = status_ptr();
    if (!status) return IX_ERR_CUDA;
    CUtensorMap tmQn{}, tmQp{};
    if (!make_query_map(&tmQn, q_nope_bf16, kNope, static_cast<uint64_t>(tokens * kH)) ||
        !make_query_map(&tmQp, q_pe_bf16, 64, static_cast<uint64_t>(tokens * kH)))
        return IX_ERR_CUDA;
    const int st = smem_setup();
    if (st != IX_OK) return st;
    SmlaArgs a{};
    a.cache = cache;
    a.num_blocks = num_blocks;
    a.block_stride = block_stride_bytes;
    a.entry_stride = entry_stride_bytes;
    a.indices = indices;
    a.tokens = tokens;
    a.block_size = block_size;
    a.topk = topk;
    a.splits = splits;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = a.ws_o + prow * kNope;
    a.status = status;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tmO{};
    if (!make_split_map(&tmO, a.ws_o, static_cast<uint64_t>(prow))) return IX_ERR_CUDA;
    smla_decode_kernel<<<static_cast<unsigned>(tokens * splits), kThreads, kSmemAlloc, s>>>(tmQn, tmQp, tmO, a);
    if (cudaGetLastError() != cudaSuccess) return IX_ERR_CUDA;
    const int64_t rows = tokens * kH;
    // the merge is the main kernel's programmatic dependent: its launch overlaps
    // the main kernel's last CTAs, and it reads the splits after pdl_wait()
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + kCombineWarps - 1) / kCombineWarps));
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, smla_combine_kernel, static_cast<const float*>(a.ws_o),
                           static_cast<const float*>(a.ws_lse), rows, splits, static_cast<uint16_t*>(out_bf16),
                           lse) != cudaSuccess)
        return IX_ERR_CUDA;
    return launch_status();
}

extern "C" int dsmla_sparse_decode_noalloc(const void* q_nope_bf16, const void* q_pe_bf16, const uint8_t* cache,
                                           int64_t num_blocks, int block_size, int64_t block_stride_bytes,
                                           int64_t entry_stride_bytes, const int32_t* indices, int64_t tokens,
                                           int heads, int topk, float sm_scale, void* out_bf16, float* lse,
                                           ix_stream_t stream) {
    // the same argument checks as dsmla_sparse_decode, in the same order; the
    // capacity check takes the place of its workspace check, before any CUDA call
    bool empty = false;
    const int chk = smla_check(q_nope_bf16, q_pe_bf16, cache, num_blocks, block_size, block_stride_bytes,
                               entry_stride_bytes, indices, tokens, heads, topk, sm_scale, out_bf16, lse, &empty);
    if (chk != IX_OK || empty) return chk;
    const int64_t splits = (static_cast<int64_t>(topk) + kSplit - 1) / kSplit;
    if (tokens > kStaticSplits || tokens * splits > kStaticSplits) return IX_ERR_WORKSPACE;
    // The scratch's device address, looked up once per device and context: a
    // context created after a reset of the device places the module (and the
    // array) anew, so the cached address is refreshed when the context changes.
    static std::mutex mu;
    struct Entry {
        void* ctx;
        void* addr;
    };
    static std::vector<Entry> cached;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IX_ERR_CUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= static_cast<int>(cached.size())) cached.resize(dev + 1, Entry{nullptr, nullptr});
        Entry& e = cached[dev];
        void* ctx = current_context();  // NULL before the runtime's first use of the device
        if (!ctx || e.ctx != ctx || !e.addr) {
            e.ctx = nullptr;
            e.addr = nullptr;
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_smla_scratch) != cudaSuccess) return IX_ERR_CUDA;
            ctx = current_context();  // the lookup has made the device's context current
            if (!ctx) return IX_ERR_CUDA;
            e.ctx = ctx;
            e.addr = p;
        }
        scratch = e.addr;
    }
    return dsmla_sparse_decode(q_nope_bf16, q_pe_bf16, cache, num_blocks, block_size, block_stride_bytes,
                               entry_stride_bytes, indices, tokens, heads, topk, sm_scale, out_bf16, lse, scratch,
                               sizeof(g_smla_scratch), stream);
}
