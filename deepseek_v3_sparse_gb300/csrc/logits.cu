// logits.cu -- FP8 MQA indexer logits on the 5th-generation tensor cores.
//
//   ix_paged_mqa_logits  decode: keys streamed from the paged indexer-K cache
//   ix_mqa_logits        prefill: keys from contiguous (gathered) K
//
// Score (DeepSeek-V3.2 lightning indexer):
//   logit[row, s] = k_scale[s] * sum_h w[row, h] * ReLU(q[row, h, :] . k[s, :])
//
// Design (one persistent CTA per SM, warp-specialised):
//   * MMA orientation: keys on M (128 per tile), (query row, head) on N.  TMEM
//     lane m then holds every head score of key m, so the weighted ReLU head
//     sum is a per-thread loop with no shuffles.
//       decode : N = 64 * next_n (the next_n rows of one request), 1 MMA job per
//                tile; TMEM holds 4 job slots of 128 columns
//       prefill: 8 query rows per group, two jobs of N = 256 (4 rows each) per
//                tile; TMEM holds 2 job slots of 256 columns.  N = 256 keeps the
//                single MMA-issuing thread at full tensor rate even while 16
//                epilogue warps compete for its SMSP's issue slots.  All 16
//                epilogue warps drain one slot while the MMAs fill the other.
//     One job = 4 x tcgen05.mma.kind::f8f6f4 (K = 128 = 4 x 32), FP32 accumulators.
//   * Warp 0 is the TMA producer: K tiles (128 B rows, 128-byte swizzle; a paged
//     tile is two 64-key blocks, each one 3-D TMA box) and per group the Q
//     operand (TMA) and head weights (bulk copy).  The epilogue reads each key's
//     fp32 scale itself (decode: from its cache block; prefill: from k_scale).
//   * Warp 1 (one elected lane) issues the MMAs and commits to mbarriers.
//   * Warps 2-17 are four epilogue warpgroups (decode: job j belongs to
//     warpgroup j % 4; prefill: warpgroup w takes row w of every job, i.e.
//     rows w and 4 + w of every group): tcgen05.ld of the accumulators, ReLU,
//     head-weighted sum (packed f32x2 FMA; the ReLU as a saturating multiply by
//     2^-25, undone exactly at the end -- decode takes half of the ReLUs as
//     FMNMX on the ALU pipe instead), key scale, masked store.  Prefill reads the accumulators in the 16x256b shape, in
//     which a thread meets only 16 heads of a row (for two keys), so its head
//     weights live in registers for the whole group and no shared-memory
//     traffic competes with the MMA operand reads; a shuffle reduce-scatter
//     finishes each key.  Decode (32x32b, one key per thread) reads its head
//     weights from shared memory.  A warp hands its slot back to the MMA warp
//     as soon as its last TMEM load has landed, before the arithmetic on that
//     chunk.
//   * The producer and MMA warps walk their loops converged and issue through
//     one lane elected once: operands computed by the whole warp stay
//     warp-uniform, which keeps the issue of a tile's four MMAs near 100 cycles.
//   * Work = the flattened list of (group, key-tile) units over all groups,
//     split evenly across CTAs on the device from context_lens / ks,ke (no host
//     sync, graph-capturable).  Each role walks the same unit sequence.
//   * Every wait is bounded (mbar_wait): on a timeout the CTA raises an abort
//     flag, all roles leave their loops, in-flight copies and MMAs are drained
//     with bounded waits, TMEM is freed, and IX_DEV_TIMEOUT is recorded.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace dsix {
namespace {

constexpr int kHeads = 64;
constexpr int kDim = 128;
constexpr int kBlk = 64;
constexpr int kTile = 128;       // keys per tile (MMA M)
constexpr int kTileBytes = kTile * kDim;
constexpr int kEpiGroups = 4;
constexpr int kThreads = 64 + kEpiGroups * 128;  // producer + MMA warps + 4 warpgroups
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstEpiWarp = 2;
constexpr int kTmemCols = 512;
constexpr uint64_t kDrainLimitNs = 100000000ull;  // 100 ms

// TK: the variant that also builds, per row, the histogram of the first radix
// digit of every logit (the ix_*_topk entry points).
template <bool kPaged, bool TK = false>
struct Cfg;

template <bool TK>
struct Cfg<true, TK> {  // decode over the paged cache
    static constexpr int kStages = 8;
    static constexpr int kSmemGroups = 2048;
    // one u32 per bin: two one-row buffers for next_n = 1, one two-row buffer for next_n = 2
    static constexpr int kHistWords = TK ? 2 * 2048 : 0;
    static constexpr int kQBytes = 2 * kHeads * kDim;  // next_n <= 2
    static constexpr int kWFloats = 2 * kHeads;
    static constexpr int kSlots = 4;
    static constexpr int kSlotCols = 128;
    static constexpr int kJobsPerTile = 1;
    static constexpr int kGroupsPerJob = 1;  // epilogue warpgroups sharing one job
};

template <bool TK>
struct Cfg<false, TK> {  // prefill over contiguous K
    static constexpr int kRows = 8;
    // the histogram variant gives up one K stage and half of the per-group
    // schedule cache to hold its 8 row histograms
    static constexpr int kStages = TK ? 3 : 4;
    static constexpr int kSmemGroups = TK ? 1024 : 2048;
    static constexpr int kHistWords = TK ? 8 * 1024 : 0;  // 8 rows, two u16 bins per word
    static constexpr int kQBytes = kRows * kHeads * kDim;  // 64 KB
    static constexpr int kWFloats = kRows * kHeads;
    static constexpr int kSlots = 2;
    static constexpr int kSlotCols = 256;
    static constexpr int kJobsPerTile = 2;   // job h covers rows 4h .. 4h + 3
    static constexpr int kGroupsPerJob = 4;  // warpgroup w takes row 4h + w of job h
    static_assert(kRows == 4 * kJobsPerTile && kGroupsPerJob == kEpiGroups, "one job row per warpgroup");
};

template <bool P, bool TK = false>
struct Smem {
    using C = Cfg<P, TK>;
    static constexpr int kQ = 0;                                     // 2 Q buffers
    static constexpr int kK = kQ + 2 * C::kQBytes;                   // K stages
    static constexpr int kW = kK + C::kStages * kTileBytes;          // 2 head-weight buffers
    static constexpr int kTiles = kW + 2 * C::kWFloats * 4;          // tiles per group
    static constexpr int kKbeg = kTiles + C::kSmemGroups * 4;         // first key of each group
    static constexpr int kHist = kKbeg + C::kSmemGroups * 4;          // row histograms (TK)
    static constexpr int kBar = kHist + C::kHistWords * 4;
    static constexpr int kNumBars = 2 * C::kStages + 4 + 2 * C::kSlots + 1 + 4;  // + 4 histogram barriers
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kScan = kMisc + 64;
    static constexpr int kTotal = kScan + 64 * 4;
    static constexpr int kAlloc = kTotal + 1024;  // slack for 1024-byte alignment
    static_assert(kAlloc <= 232448, "shared memory budget");
    static_assert(kK % 1024 == 0 && C::kQBytes % 1024 == 0, "128-byte-swizzled TMA tiles: 1024 B");
    static_assert(kW % 16 == 0 && kBar % 8 == 0, "alignment");
};

struct LogitsArgs {
    const float* w;
    float* logits;
    int64_t ld;
    int num_groups;
    int* status;
    // decode
    const int32_t* context_lens;
    const int32_t* bt;
    const uint8_t* cache;  // the paged cache (key scales are read from it directly)
    int64_t bt_stride;
    int next_n;
    int64_t num_blocks;
    // prefill
    const float* k_scale;
    const int32_t* ks;
    const int32_t* ke;
    int64_t tq;
    int64_t tk;
};

// Kernel arguments beyond LogitsArgs (an argument of their own: widening
// LogitsArgs costs the plain kernels registers).
//   hist, k     histogram variant: rows with more than k visible keys add the
//               first radix digit of each of their logits to
//               hist[row * kHistRowWords ...]
//   group_cost  the schedule's cost of a group beyond its tiles, in tiles: the
//               work of each CTA is (tiles + group_cost per group started)
//               split evenly, so CTAs that meet many short groups (the first
//               rows of a causal chunk) get fewer tiles
struct HistArgs {
    uint32_t* hist;
    int k;
    int group_cost;
};

// Group costs of the schedule (tiles), measured per kernel kind.
constexpr int kGroupCostPrefill = 2;
constexpr int kGroupCostDecode = 0;

// ---------------------------------------------------------------------------
// per-row visible ranges (clamped; report=true records why)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int decode_row_len(const LogitsArgs& a, int ctx, int j, bool report) {
    int64_t L = static_cast<int64_t>(ctx) - a.next_n + 1 + j;
    if (L < 0) L = 0;
    if (L > a.ld) {
        if (report) flag(a.status, IX_DEV_ROW_TOO_LONG);
        L = a.ld;
    }
    return static_cast<int>(L);
}

__device__ __forceinline__ void prefill_row_range(const LogitsArgs& a, int64_t r, int& s0, int& s1,
                                                  bool report) {
    int64_t x0 = __ldg(a.ks + r), x1 = __ldg(a.ke + r);
    if (x0 < 0 || x1 > a.tk || x1 < x0) {
        if (report) flag(a.status, IX_DEV_BAD_RANGE);
        x0 = x0 < 0 ? 0 : x0;
        x1 = x1 > a.tk ? a.tk : x1;
        if (x1 < x0) x1 = x0;
    }
    if (x1 - x0 > a.ld) {
        if (report) flag(a.status, IX_DEV_ROW_TOO_LONG);
        x1 = x0 + a.ld;
    }
    s0 = static_cast<int>(x0);
    s1 = static_cast<int>(x1);
}

// Key range [kbeg, kend) that a group's rows need.
template <bool P>
__device__ __forceinline__ void group_range(const LogitsArgs& a, int g, int& kbeg, int& kend,
                                            bool report) {
    if constexpr (P) {
        kbeg = 0;
        kend = decode_row_len(a, __ldg(a.context_lens + g), a.next_n - 1, report);
    } else {
        kbeg = 0x7fffffff;
        kend = 0;
        const int64_t r0 = static_cast<int64_t>(g) * Cfg<false>::kRows;
#pragma unroll
        for (int i = 0; i < Cfg<false>::kRows; ++i) {
            if (r0 + i >= a.tq) break;
            int s0, s1;
            prefill_row_range(a, r0 + i, s0, s1, report);
            if (s1 > s0) {
                kbeg = min(kbeg, s0);
                kend = max(kend, s1);
            }
        }
        if (kend == 0) kbeg = 0;
    }
}

template <bool P>
__device__ __forceinline__ int group_tiles(const LogitsArgs& a, int g, bool report) {
    int kb, ke;
    group_range<P>(a, g, kb, ke, report);
    return ke > kb ? (ke - kb + kTile - 1) / kTile : 0;
}

// Block-wide exclusive scan of one int per thread; *total receives the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        constexpr int nw = kThreads / 32;
        int s = lane < nw ? scratch[lane] : 0;
        int inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < nw) scratch[32 + lane] = inc - s;
        if (lane == nw - 1) scratch[63] = inc;
    }
    __syncthreads();
    const int r = scratch[32 + warp] + x - v;
    *total = scratch[63];
    __syncthreads();
    return r;
}

// Walks the flattened (group, tile) units of this CTA.  Groups below CAP
// have their tile counts cached in shared memory.
template <bool P, int CAP>
struct Cursor {
    int g, t, ntiles, left;
    __device__ __forceinline__ int tiles_of(const LogitsArgs& a, const int* s_tiles, int gg) const {
        if (gg >= a.num_groups) return 0;
        return gg < CAP ? s_tiles[gg] : group_tiles<P>(a, gg, false);
    }
    // Returns true when the next unit starts a new group.  Never walks past
    // the last group: if the unit count and the groups disagree, it stops.
    __device__ __forceinline__ bool advance(const LogitsArgs& a, const int* s_tiles) {
        ++t;
        --left;
        if (left > 0 && t >= ntiles) {
            do {
                ++g;
                ntiles = tiles_of(a, s_tiles, g);
            } while (ntiles == 0 && g < a.num_groups);
            t = 0;
            if (g >= a.num_groups) left = 0;
            return true;
        }
        return false;
    }
};

__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag (drains in-flight work on the way out);
// `never` points at a shared-memory word that stays 0.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, volatile int* never,
                                           int* status) {
    mbar_wait(bar, parity, never, status, kDrainLimitNs);
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// max(s, 0) * 2^-25 in one saturating multiply on the FMA pipe.  Exact: the
// product is a power-of-two scaling, and |s| < 2^25 for any score of e4m3
// operands (|q . k| <= 128 * 448^2), so saturation at 1 never clips a score.
__device__ __forceinline__ float relu_scaled(float s) {
    float r;
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(s), "f"(0x1p-25f));
    return r;
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Head-weighted ReLU sums for this thread's key over R query rows: TMEM
// columns [tbase + 64 r, +64) hold row r's 64 head scores, w[64 r + h] the
// row's head weights.  The load of 32-column chunk c+1 overlaps the
// arithmetic on chunk c; `release` runs once the last chunk is in registers
// (the TMEM columns may then be overwritten).  Heads are taken in pairs: the
// even head's ReLU is an FMNMX (ALU pipe), the odd head's a saturating
// multiply by 2^-25 (FMA pipe), and one packed f32x2 FMA accumulates both; the
// odd-head lane is rescaled by 2^25 (exactly) at the end.
template <int R, class Release>
__device__ __forceinline__ void head_sums(uint32_t tbase, const float* w, float (&out)[R], Release&& release) {
    uint32_t buf[2][32];
    uint64_t acc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0ull;
    tmem_ld32(tbase, buf[0]);
    tmem_wait_ld(buf[0]);
#pragma unroll
    for (int c = 0; c < 2 * R; ++c) {
        if (c + 1 < 2 * R) tmem_ld32(tbase + (c + 1) * 32, buf[(c + 1) & 1]);
        const int r = c >> 1;
        const float4* w4 = reinterpret_cast<const float4*>(w + r * kHeads + (c & 1) * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 ww = w4[q];
            const uint32_t* v = buf[c & 1] + 4 * q;
            const uint64_t t01 =
                pack2(fmaxf(__uint_as_float(v[0]), 0.f), relu_scaled(__uint_as_float(v[1])));
            const uint64_t t23 =
                pack2(fmaxf(__uint_as_float(v[2]), 0.f), relu_scaled(__uint_as_float(v[3])));
            acc[r][0] = fma2(pack2(ww.x, ww.y), t01, acc[r][0]);
            acc[r][1] = fma2(pack2(ww.z, ww.w), t23, acc[r][1]);
        }
        if (c + 1 < 2 * R) {
            tmem_wait_ld(buf[(c + 1) & 1]);
            if (c + 2 == 2 * R) release();
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        float e0, o0, e1, o1;
        unpack2(acc[r][0], e0, o0);
        unpack2(acc[r][1], e1, o1);
        out[r] = (e0 + e1) + (o0 + o1) * 0x1p25f;
    }
}

// Prefill head sum of one query row for the 32 keys of a warp's TMEM lane
// quadrant, read in the 16x256b shape: for each 16-lane half, thread t holds
// keys t/4 and t/4 + 8 of the half for heads 8j + 2(t%4) + {0, 1}, j = 0..7.  A
// thread therefore needs only 16 of the row's head weights (w2[j] = the packed
// pair for repeat j), which stay in registers for a whole group.  Four chunks
// of 32 columns, (half 0, heads 0-31), (half 0, heads 32-63), (half 1, ...),
// each in flight while the previous one is summed; `release` runs once the last
// chunk is in registers.  The four threads t%4 = 0..3 that hold a key's partial
// sums combine them in a two-step reduce-scatter: thread t returns the total of
// key (16 ((t%4) >> 1) + 8 ((t%4) & 1) + t/4) of the quadrant.
template <class Release>
__device__ __forceinline__ float head_sums_16x256b(uint32_t tbase, const uint64_t (&w2)[8], int tq,
                                                   Release&& release) {
    uint32_t buf[2][16];
    float part[4];  // (half 0, key a), (half 0, key b), (half 1, key a), (half 1, key b)
    uint64_t acc[2];  // keys a and b of the current half: (even heads, odd heads), both scaled by 2^-25
    tmem_ld16x256b_x4(tbase, buf[0]);
    tmem_wait_ld(buf[0]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int half = c >> 1, cc = c & 1;
        if (c + 1 < 4) {
            const int nh = (c + 1) >> 1, ncc = (c + 1) & 1;
            tmem_ld16x256b_x4(tbase + (static_cast<uint32_t>(16 * nh) << 16) + 32 * ncc, buf[(c + 1) & 1]);
        }
        if (cc == 0) acc[0] = acc[1] = 0ull;
        const uint32_t* v = buf[c & 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint64_t wp = w2[4 * cc + j];
            // both ReLUs as saturating multiplies by 2^-25 (the FMA pipe measured
            // faster here than splitting them with FMNMX on the ALU pipe)
            const uint64_t ta = pack2(relu_scaled(__uint_as_float(v[4 * j])), relu_scaled(__uint_as_float(v[4 * j + 1])));
            const uint64_t tb =
                pack2(relu_scaled(__uint_as_float(v[4 * j + 2])), relu_scaled(__uint_as_float(v[4 * j + 3])));
            acc[0] = fma2(wp, ta, acc[0]);
            acc[1] = fma2(wp, tb, acc[1]);
        }
        if (cc == 1) {  // still scaled by 2^-25; undone once after the reduction
            float e, o;
            unpack2(acc[0], e, o);
            part[2 * half] = e + o;
            unpack2(acc[1], e, o);
            part[2 * half + 1] = e + o;
        }
        if (c + 1 < 4) {
            tmem_wait_ld(buf[(c + 1) & 1]);
            if (c + 2 == 4) release();
        }
    }
    // reduce-scatter over the 4 threads of a key: first across halves (lane ^ 2),
    // then across keys a / b (lane ^ 1)
    const bool hi = (tq & 2) != 0, odd = (tq & 1) != 0;
    const float s0 = __shfl_xor_sync(0xffffffffu, hi ? part[0] : part[2], 2);
    const float s1 = __shfl_xor_sync(0xffffffffu, hi ? part[1] : part[3], 2);
    const float x0 = (hi ? part[2] : part[0]) + s0;
    const float x1 = (hi ? part[3] : part[1]) + s1;
    const float r = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
    return ((odd ? x1 : x0) + r) * 0x1p25f;  // undo the ReLU's 2^-25 (exact)
}

template <bool P, int NN, bool TK>
__global__ void __launch_bounds__(kThreads, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmQ,
                  const LogitsArgs a, const HistArgs hk) {
    using C = Cfg<P, TK>;
    using S = Smem<P, TK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = sm + S::kQ;
    uint8_t* sK = sm + S::kK;
    float* sW = reinterpret_cast<float*>(sm + S::kW);
    int* s_tiles = reinterpret_cast<int*>(sm + S::kTiles);
    int* s_kbeg = reinterpret_cast<int*>(sm + S::kKbeg);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + S::kBar);
    uint64_t* empty = full + C::kStages;
    uint64_t* qw_full = empty + C::kStages;
    uint64_t* qw_empty = qw_full + 2;
    uint64_t* acc_full = qw_empty + 2;
    uint64_t* acc_empty = acc_full + C::kSlots;
    uint64_t* mma_done = acc_empty + C::kSlots;
    uint64_t* hbar = mma_done + 1;  // histogram hand-offs (TK): one per warpgroup (prefill); decode: filled [0..1], cleared [2..3]
    uint32_t* s_hist = reinterpret_cast<uint32_t*>(sm + S::kHist);
    int* misc = reinterpret_cast<int*>(sm + S::kMisc);  // tmem base, abort, g0, t0, units
    int* scan = reinterpret_cast<int*>(sm + S::kScan);
    volatile int* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qw_full + i, 1);
            mbar_init(qw_empty + i, 4 * kEpiGroups);
        }
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, 4 * C::kGroupsPerJob);
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < 4; ++i) mbar_init(hbar + i, P ? 4 * kEpiGroups : 4);
        fence_barrier_init();
        misc[1] = 0;
        misc[4] = 0;
        misc[5] = 0;  // never raised: the abort flag seen by drain waits
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmQ);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(reinterpret_cast<uint32_t*>(misc), kTmemCols);
        tmem_relinquish();
    }
    if constexpr (TK) {
        for (int i = threadIdx.x; i < C::kHistWords; i += kThreads) s_hist[i] = 0u;
    }

    // ---- schedule: split the flattened unit list evenly across CTAs ----
    const int G = a.num_groups;
    int local = 0;
    for (int g = threadIdx.x; g < G; g += kThreads) {
        int kb, ke;
        group_range<P>(a, g, kb, ke, blockIdx.x == 0);
        const int n = ke > kb ? (ke - kb + kTile - 1) / kTile : 0;
        if (g < C::kSmemGroups) {
            s_tiles[g] = n;
            s_kbeg[g] = kb;
        }
        local += n;
    }
    // Weighted split: group g costs n(g) + gc tiles of work (gc for a group
    // with tiles), CTA c takes the weighted range [c W / grid, (c+1) W / grid),
    // and a weighted position x inside group g maps to its real tile
    // min(n(g), max(0, x - ws(g) - gc)) (the group's overhead comes first).
    // u0 / u1 are the CTA's real tile range in the flattened tile list.
    const int gc = hk.group_cost;
    int U;
    const int excl0 = block_excl_scan(local, scan, &U);
    int64_t u0, u1;
    if (gc == 0) {
        u0 = static_cast<int64_t>(blockIdx.x) * U / gridDim.x;
        u1 = static_cast<int64_t>(blockIdx.x + 1) * U / gridDim.x;
    } else {
        // weighted costs of this thread's groups, and their total
        int wlocal = 0;
        for (int g = threadIdx.x; g < G; g += kThreads) {
            const int n = g < C::kSmemGroups ? s_tiles[g] : group_tiles<P>(a, g, false);
            wlocal += n > 0 ? n + gc : 0;
        }
        int W;
        block_excl_scan(wlocal, scan, &W);
        const int64_t w0 = static_cast<int64_t>(blockIdx.x) * W / gridDim.x;
        const int64_t w1 = static_cast<int64_t>(blockIdx.x + 1) * W / gridDim.x;
        if (threadIdx.x == 0) {
            misc[6] = U;  // real positions of w0 / w1; W maps to U
            misc[7] = U;
        }
        __syncthreads();
        int wrun = 0, rrun = 0;
        for (int base = 0; base < G && (wrun <= w0 || wrun <= w1); base += kThreads) {
            const int g = base + threadIdx.x;
            const int n = g < G ? (g < C::kSmemGroups ? s_tiles[g] : group_tiles<P>(a, g, false)) : 0;
            const int wc = n > 0 ? n + gc : 0;
            int wchunk, rchunk;
            const int ws = block_excl_scan(wc, scan, &wchunk) + wrun;
            const int rs = block_excl_scan(n, scan, &rchunk) + rrun;
            if (wc > 0 && ws <= w0 && w0 < ws + wc) {
                const int64_t x = w0 - ws - gc;
                misc[6] = rs + static_cast<int>(x < 0 ? 0 : (x > n ? n : x));
            }
            if (wc > 0 && ws <= w1 && w1 < ws + wc) {
                const int64_t x = w1 - ws - gc;
                misc[7] = rs + static_cast<int>(x < 0 ? 0 : (x > n ? n : x));
            }
            wrun += wchunk;
            rrun += rchunk;
        }
        __syncthreads();
        u0 = misc[6];
        u1 = misc[7];
        __syncthreads();  // misc[6..7] are not rewritten, but misc[2..4] are written below
    }
    if (G <= kThreads) {
        // one group per thread: the scan above already placed every group
        if (u1 > u0 && local > 0 && excl0 <= u0 && u0 < excl0 + local) {
            misc[2] = threadIdx.x;
            misc[3] = static_cast<int>(u0 - excl0);
            misc[4] = static_cast<int>(u1 - u0);
        }
    } else if (u1 > u0) {
        int running = 0;
        for (int base = 0; base < G && running <= u0; base += kThreads) {
            const int g = base + threadIdx.x;
            const int n = g < G ? (g < C::kSmemGroups ? s_tiles[g] : group_tiles<P>(a, g, false)) : 0;
            int chunk;
            const int excl = block_excl_scan(n, scan, &chunk) + running;
            if (n > 0 && excl <= u0 && u0 < excl + n) {
                misc[2] = g;
                misc[3] = static_cast<int>(u0 - excl);
                misc[4] = static_cast<int>(u1 - u0);
            }
            running += chunk;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = static_cast<uint32_t>(misc[0]);
    const int units = misc[4];
    // key range of a group; prefill groups' first keys were kept in shared
    // memory by the schedule (their end is not needed past it)
    auto group_bounds = [&](int gg, int& kb, int& ke) {
        if (!P && gg < C::kSmemGroups) {
            kb = s_kbeg[gg];
            ke = 0;
        } else {
            group_range<P>(a, gg, kb, ke, false);
        }
    };

    if (units > 0) {
        Cursor<P, C::kSmemGroups> cur;
        cur.g = misc[2];
        cur.t = misc[3];
        cur.left = units;
        cur.ntiles = cur.tiles_of(a, s_tiles, cur.g);

        if (warp == kProducerWarp) {
            // ------------------------------------------------------------ producer
            // The whole warp walks the loop; one lane, elected once, issues the copies.
            // Paged K tiles are read once per launch: they go through L2 as
            // evict-first lines, so the stream does not force out (and write back)
            // lines that earlier work left dirty there.
            const bool leader = elect_one();
            const uint64_t stream_policy = P ? l2_evict_first_policy() : 0;
            int it = 0, qi = 0;
            int kbeg = 0, kend = 0;
            // decode: lane l holds the block-table entry of block 2 * bt_base + l (16
            // tiles); the next window of the group is loaded one window ahead
            int bt_base = -1, bt_val = -1, bt_nxt = -1;
            auto bt_fetch = [&](int gg, int t0) {
                const int bi = 2 * t0 + lane;
                return bi * kBlk < kend ? __ldg(a.bt + static_cast<int64_t>(gg) * a.bt_stride + bi) : -1;
            };
            bool new_group = true;
            while (cur.left > 0) {
                const int g = cur.g;
                if (new_group) {
                    group_bounds(g, kbeg, kend);
                    bt_base = -1;
                    const int qb = qi & 1;
                    if (!wait_warp(qw_empty + qb, ((qi >> 1) & 1) ^ 1, abort_flag, a.status)) break;
                    if (leader) {
                        uint8_t* qdst = sQ + qb * C::kQBytes;
                        float* wdst = sW + qb * C::kWFloats;
                        if constexpr (P) {
                            const uint32_t wbytes = a.next_n * kHeads * 4;
                            mbar_arrive_expect_tx(qw_full + qb, a.next_n * kHeads * kDim + wbytes);
                            tma_load_2d(qdst, &tmQ, qw_full + qb, 0, g * a.next_n * kHeads);
                            bulk_load(wdst, a.w + static_cast<int64_t>(g) * a.next_n * kHeads, wbytes,
                                      qw_full + qb);
                        } else {
                            const int64_t r0 = static_cast<int64_t>(g) * C::kRows;
                            const int nrows = static_cast<int>(a.tq - r0 < C::kRows ? a.tq - r0 : C::kRows);
                            const uint32_t wbytes = nrows * kHeads * 4;
                            mbar_arrive_expect_tx(qw_full + qb, C::kQBytes + wbytes);
                            const int qrow = static_cast<int>(r0 * kHeads);
                            tma_load_2d(qdst, &tmQ, qw_full + qb, 0, qrow);
                            tma_load_2d(qdst + C::kQBytes / 2, &tmQ, qw_full + qb, 0, qrow + 256);
                            bulk_load(wdst, a.w + r0 * kHeads, wbytes, qw_full + qb);
                        }
                    }
                    ++qi;
                }
                const int stage = it % C::kStages;
                if (!wait_warp(empty + stage, ((it / C::kStages) & 1) ^ 1, abort_flag, a.status)) break;
                uint8_t* kdst = sK + stage * kTileBytes;
                if constexpr (P) {
                    if (bt_base < 0 || cur.t - bt_base >= 16) {
                        const int raw = (bt_base >= 0 && cur.t == bt_base + 16) ? bt_nxt : bt_fetch(g, cur.t);
                        bt_base = cur.t;
                        bt_nxt = bt_fetch(g, bt_base + 16);
                        bt_val = -1;
                        if ((2 * bt_base + lane) * kBlk < kend) {
                            bt_val = raw;
                            if (bt_val < 0 || bt_val >= a.num_blocks) {
                                flag(a.status, IX_DEV_BAD_BLOCK);
                                bt_val = static_cast<int>(a.num_blocks);  // out of the map: zero fill
                            }
                        }
                    }
                    const int blk0 = __shfl_sync(0xffffffffu, bt_val, 2 * (cur.t - bt_base));
                    const int blk1 = __shfl_sync(0xffffffffu, bt_val, 2 * (cur.t - bt_base) + 1);
                    const bool two = (2 * cur.t + 1) * kBlk < kend;
                    if (leader) {
                        mbar_arrive_expect_tx(full + stage, two ? kTileBytes : kTileBytes / 2);
                        tma_load_3d_hint(kdst, &tmK, full + stage, 0, 0, blk0, stream_policy);
                        if (two) tma_load_3d_hint(kdst + kTileBytes / 2, &tmK, full + stage, 0, 0, blk1, stream_policy);
                    }
                } else {
                    const int start = kbeg + cur.t * kTile;
                    if (leader) {
                        mbar_arrive_expect_tx(full + stage, kTileBytes);
                        tma_load_2d(kdst, &tmK, full + stage, 0, start);
                    }
                }
                ++it;
                new_group = cur.advance(a, s_tiles);
            }
            // drain: the last copies issued into each buffer must land before exit
            if (lane == 0) {
                for (int i = max(0, it - C::kStages); i < it; ++i)
                    drain_wait(full + i % C::kStages, (i / C::kStages) & 1, misc + 5, a.status);
                for (int i = max(0, qi - 2); i < qi; ++i)
                    drain_wait(qw_full + (i & 1), (i >> 1) & 1, misc + 5, a.status);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // The whole warp walks the loop and waits; one lane, elected once, issues
            // every MMA and commit (a commit tracks the issuing thread's MMAs), so
            // every operand stays warp-uniform.
            const bool leader = elect_one();
            int it = 0, qi = 0, job = 0;
            uint64_t qdesc = 0;
            bool issued = false, new_group = true;
            constexpr int kJobN = P ? kHeads * NN : kHeads * 4;
            constexpr uint32_t idesc = idesc_e4m3_f32(kTile, kJobN);
            // descriptors advance by (bytes >> 4) in the start-address field
            const uint64_t a_desc0 = sdesc_k_sw128(smem_u32(sK));
            while (cur.left > 0) {
                if (new_group) {
                    const int qb = qi & 1;
                    if (!wait_warp(qw_full + qb, (qi >> 1) & 1, abort_flag, a.status)) break;
                    qdesc = sdesc_k_sw128(smem_u32(sQ + qb * C::kQBytes));
                    ++qi;
                }
                const int stage = it % C::kStages;
                if (!wait_warp(full + stage, (it / C::kStages) & 1, abort_flag, a.status)) break;
                tc_fence_after();
                const uint64_t adesc = a_desc0 + static_cast<uint64_t>(stage * (kTileBytes >> 4));
                bool ok = true;
#pragma unroll
                for (int h = 0; h < C::kJobsPerTile; ++h) {
                    const int slot = job % C::kSlots;
                    if (!wait_warp(acc_empty + slot, ((job / C::kSlots) & 1) ^ 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + slot * C::kSlotCols;
                    const uint64_t bdesc = qdesc + static_cast<uint64_t>(h * ((kJobN * kDim) >> 4));
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kDim / 32; ++kk)
                            mma_e4m3(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, kk > 0);
                        mma_commit(acc_full + slot);
                    }
                    __syncwarp();
                    issued = true;
                    ++job;
                }
                if (!ok) break;
                if (leader) mma_commit(empty + stage);
                __syncwarp();
                ++it;
                new_group = cur.advance(a, s_tiles);
            }
            if (issued) {
                if (leader) {
                    mma_commit(mma_done);
                    drain_wait(mma_done, 0, misc + 5, a.status);
                }
                __syncwarp();
            }
        } else if constexpr (!P) {
            // ------------------------------------------------------------ prefill epilogue
            // Warpgroup wg sums rows wg (job 0) and 4 + wg (job 1) of every group; the
            // accumulators are read in the 16x256b shape (head_sums_16x256b), so each
            // thread keeps the 16 head weights it needs of each of its two rows in
            // registers for the whole group.
            const int wg = (warp - kFirstEpiWarp) >> 2;
            const int quad = warp & 3;
            const int tq = lane & 3;
            const int m = quad * 32 + 16 * (tq >> 1) + 8 * (tq & 1) + (lane >> 2);  // key this thread stores
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
            int qi = 0, job = 0;
            int kbeg = 0, kend = 0;
            int rs0[2], rs1[2];  // visible key range of rows wg and 4 + wg
            float* orow[2];      // their logits rows
            uint64_t w2[2][8];   // packed head-weight pairs of those rows
            bool new_group = true, have_group = false, live = true;
            // TK: the warpgroup's two rows keep their digit histograms in shared
            // memory (two u16 counters per word); a hand-off adds them to the
            // rows' global histograms and clears them.  It runs when the group
            // ends, and every 256 tiles of one group so no u16 counter overflows.
            bool hw0 = false, hw1 = false;  // rows wg and 4 + wg have more than k keys
            int64_t hr0 = 0, hr1 = 0;       // their row indices
            uint32_t hsync = 0;             // waits done on this warpgroup's hand-off barrier
            int gtiles = 0;                 // tiles of the current group since the last hand-off
            auto hflush = [&]() -> bool {
                __syncwarp();
                if (lane == 0) mbar_arrive(hbar + wg);
                if (!wait_warp(hbar + wg, hsync & 1, abort_flag, a.status)) return false;
                ++hsync;
                // warp `quad` of the warpgroup takes words [512 quad, 512 quad + 512) of
                // its 2 x 1024 words, 16 per lane: 32 fine bins = one coarse bin
                const int w0 = 512 * quad + 16 * lane;
                const int hh = w0 >> 10, wr = w0 & 1023;
                uint4* src = reinterpret_cast<uint4*>(s_hist + (4 * hh + wg) * 1024 + wr);
                uint32_t x[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = src[i];
                    x[4 * i] = v.x;
                    x[4 * i + 1] = v.y;
                    x[4 * i + 2] = v.z;
                    x[4 * i + 3] = v.w;
                    src[i] = make_uint4(0u, 0u, 0u, 0u);
                }
                if (hh ? hw1 : hw0) {
                    uint32_t* G = hk.hist + (hh ? hr1 : hr0) * kHistRowWords;
                    uint32_t csum = 0;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t lo = x[i] & 0xFFFFu, hi = x[i] >> 16;
                        if (lo) atomicAdd(G + kHistCoarse + 2 * (wr + i), lo);
                        if (hi) atomicAdd(G + kHistCoarse + 2 * (wr + i) + 1, hi);
                        csum += lo + hi;
                    }
                    if (csum) atomicAdd(G + (wr >> 4), csum);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(hbar + wg);
                if (!wait_warp(hbar + wg, hsync & 1, abort_flag, a.status)) return false;
                ++hsync;
                return true;
            };
            while (cur.left > 0) {
                const int g = cur.g;
                if (new_group) {
                    if constexpr (TK) {
                        if (have_group && !hflush()) {
                            live = false;
                            break;
                        }
                        gtiles = 0;
                    }
                    if (have_group) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(qw_empty + ((qi - 1) & 1));
                    }
                    if (!wait_warp(qw_full + (qi & 1), (qi >> 1) & 1, abort_flag, a.status)) {
                        live = false;
                        break;
                    }
                    have_group = true;
                    group_bounds(g, kbeg, kend);
                    const float* wq = sW + (qi & 1) * C::kWFloats;
                    ++qi;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int64_t r = static_cast<int64_t>(g) * C::kRows + 4 * h + wg;
                        rs0[h] = 0;
                        rs1[h] = 0;
                        if (r < a.tq) prefill_row_range(a, r, rs0[h], rs1[h], false);
                        orow[h] = a.logits + (r < a.tq ? r : 0) * a.ld;
                        const float* wr = wq + (4 * h + wg) * kHeads + 2 * tq;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float2 wv = *reinterpret_cast<const float2*>(wr + 8 * j);
                            w2[h][j] = pack2(wv.x, wv.y);
                        }
                    }
                    if constexpr (TK) {
                        hr0 = static_cast<int64_t>(g) * C::kRows + wg;
                        hr1 = hr0 + 4;
                        hw0 = hr0 < a.tq && rs1[0] - rs0[0] > hk.k;
                        hw1 = hr1 < a.tq && rs1[1] - rs0[1] > hk.k;
                    }
                }
                const int s = kbeg + cur.t * kTile + m;  // key index
                // the scale comes straight from L2, issued before the waits
                const float ksc = __ldg(a.k_scale + min(static_cast<int64_t>(s), a.tk - 1));
                bool ok = true;
#pragma unroll
                for (int h = 0; h < C::kJobsPerTile; ++h, ++job) {
                    const int slot = job % C::kSlots;
                    if (!wait_warp(acc_full + slot, (job / C::kSlots) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float sum =
                        head_sums_16x256b(lane_addr + slot * C::kSlotCols + wg * kHeads, w2[h], tq, [&] {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(acc_empty + slot);
                        });
                    if (s >= rs0[h] && s < rs1[h]) {
                        const float v = sum * ksc;
                        orow[h][s - rs0[h]] = v;
                        if constexpr (TK) {
                            if (h ? hw1 : hw0) {
                                const uint32_t d = order_key(v) >> kDigitShift;
                                atomicAdd(s_hist + (4 * h + wg) * 1024 + (d >> 1), 1u << ((d & 1u) << 4));
                            }
                        }
                    }
                }
                if (!ok) {
                    live = false;
                    break;
                }
                new_group = cur.advance(a, s_tiles);
                if constexpr (TK) {
                    if (!new_group && cur.left > 0 && ++gtiles == 256) {  // long rows: keep the u16 counters small
                        gtiles = 0;
                        if (!hflush()) {
                            live = false;
                            break;
                        }
                    }
                }
            }
            if constexpr (TK) {
                if (live && have_group) hflush();
            }
        } else {
            // ------------------------------------------------------------ decode epilogue
            // Job j (tile j of this CTA) belongs to warpgroup j % 4; each thread sums the
            // next_n rows of its key.
            const int wg = (warp - kFirstEpiWarp) >> 2;
            const int quad = warp & 3;
            const int m = quad * 32 + lane;  // tile row = TMEM lane
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
            int qi = 0, job = 0;
            int kbeg = 0, kend = 0;
            int rs1[NN];  // visible length of each row of the group
            bool new_group = true, have_group = false, live = true;
            // TK: the group's rows keep one u32 digit histogram each in shared
            // memory, shared by all 16 epilogue warps (jobs rotate over the
            // warpgroups).  A warp leaving a group arrives on its buffer's
            // "filled" barrier; once all 16 have, each warp adds its share of the
            // buffer to the rows' global histograms, clears it and arrives on the
            // buffer's "cleared" barrier, which a warp waits on before it counts
            // into that buffer for a later group.  One-row groups alternate
            // between two buffers and defer the flush (a warp runs it as soon as
            // it finds the filled barrier complete at a later unit, at the latest
            // when it leaves the next group), so with groups of more than a few
            // tiles no warp stops at a group change.  Two-row groups fill the one
            // buffer the space holds and flush it when they leave the group
            // (measured faster there than a second buffer would be).
            constexpr int kHB = NN == 1 ? 2 : 1;  // histogram buffers
            uint64_t* hfill = hbar;     // [2]
            uint64_t* hclr = hbar + 2;  // [2]
            uint32_t hwm0 = 0, hwm1 = 0;  // per buffer: bit j set when row j has more than k keys
            int hr0 = 0, hr1 = 0;         // per buffer: first row of its group
            int huse0 = 0, huse1 = 0;     // per buffer: groups that have counted into it
            int hb = 0;                   // buffer of the current group
            int pend = -1;                // buffer all warps have filled, not yet flushed by this warp
            auto flush_share = [&](int b) {
                const int et = threadIdx.x - kFirstEpiWarp * 32;  // 0..511: fine bins 4 et .. 4 et + 3
                const uint32_t wm = b ? hwm1 : hwm0;
                const int64_t row0 = b ? hr1 : hr0;  // rows fit in int: a row's logits start at row * ld
#pragma unroll
                for (int j = 0; j < NN; ++j) {
                    uint4* src = reinterpret_cast<uint4*>(s_hist + (NN * b + j) * kHistFine + 4 * et);
                    const uint4 v = *src;
                    *src = make_uint4(0u, 0u, 0u, 0u);
                    if ((wm >> j) & 1u) {  // uniform over the CTA
                        uint32_t* G = hk.hist + (row0 + j) * kHistRowWords;
                        if (v.x) atomicAdd(G + kHistCoarse + 4 * et, v.x);
                        if (v.y) atomicAdd(G + kHistCoarse + 4 * et + 1, v.y);
                        if (v.z) atomicAdd(G + kHistCoarse + 4 * et + 2, v.z);
                        if (v.w) atomicAdd(G + kHistCoarse + 4 * et + 3, v.w);
                        uint32_t csum = (v.x + v.y) + (v.z + v.w);  // a coarse bin = 8 consecutive threads
                        csum += __shfl_xor_sync(0xffffffffu, csum, 1);
                        csum += __shfl_xor_sync(0xffffffffu, csum, 2);
                        csum += __shfl_xor_sync(0xffffffffu, csum, 4);
                        if ((lane & 7) == 0 && csum) atomicAdd(G + (et >> 3), csum);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(hclr + b);
            };
            // the pending buffer's flush; `block` waits for its filled barrier,
            // otherwise the flush runs only if that barrier is already complete
            auto flush_pending = [&](bool block) -> bool {
                if (pend < 0) return true;
                const uint32_t ph = static_cast<uint32_t>((pend ? huse1 : huse0) - 1) & 1u;
                if (block) {
                    if (!wait_warp(hfill + pend, ph, abort_flag, a.status)) return false;
                } else if (!__all_sync(0xffffffffu, mbar_try_wait(hfill + pend, ph))) {
                    return true;
                }
                flush_share(pend);
                pend = -1;
                return true;
            };
            while (cur.left > 0) {
                const int g = cur.g;
                if (new_group) {
                    if constexpr (TK) {
                        if (have_group) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(hfill + hb);  // this warp's counts of the group are in
                            if (!flush_pending(true)) {  // the buffer before, if this warp has not flushed it yet
                                live = false;
                                break;
                            }
                            pend = hb;
                            if constexpr (kHB == 2) hb ^= 1;
                            if (kHB == 1 && !flush_pending(true)) {
                                live = false;
                                break;
                            }
                        }
                        const int used = hb ? huse1 : huse0;
                        if (used > 0 && !wait_warp(hclr + hb, static_cast<uint32_t>(used - 1) & 1u, abort_flag, a.status)) {
                            live = false;
                            break;
                        }
                        if (hb) ++huse1; else ++huse0;
                    }
                    if (have_group) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(qw_empty + ((qi - 1) & 1));
                    }
                    if (!wait_warp(qw_full + (qi & 1), (qi >> 1) & 1, abort_flag, a.status)) {
                        live = false;
                        break;
                    }
                    ++qi;
                    have_group = true;
                    group_bounds(g, kbeg, kend);
                    const int ctx = __ldg(a.context_lens + g);
#pragma unroll
                    for (int j = 0; j < NN; ++j) rs1[j] = decode_row_len(a, ctx, j, false);
                    if constexpr (TK) {
                        uint32_t wm = 0;
#pragma unroll
                        for (int j = 0; j < NN; ++j) wm |= (rs1[j] > hk.k ? 1u : 0u) << j;
                        if (hb) {
                            hwm1 = wm;
                            hr1 = g * NN;
                        } else {
                            hwm0 = wm;
                            hr0 = g * NN;
                        }
                    }
                } else if constexpr (TK) {
                    if (pend >= 0 && !flush_pending(false)) {
                        live = false;
                        break;
                    }
                }
                const float* wq = sW + ((qi - 1) & 1) * C::kWFloats;
                const int s = kbeg + cur.t * kTile + m;  // key index
                bool ok = true;
                if ((job & 3) == wg) {
                    const int slot = job % C::kSlots;
                    // the key's scale straight from its cache block (a warp's 32 keys share
                    // one block-table entry), issued before the accumulator wait and used
                    // only at the store; invalid blocks read as scale 0 like the
                    // zero-filled tile the producer loads for them
                    float ksc = 0.f;
                    if (s < kend) {
                        const int blk = __ldg(a.bt + static_cast<int64_t>(g) * a.bt_stride + (s >> 6));
                        if (blk >= 0 && blk < a.num_blocks)
                            ksc = __ldg(reinterpret_cast<const float*>(
                                            a.cache + static_cast<int64_t>(blk) * (kBlk * (kDim + 4)) + kBlk * kDim) +
                                        (s & (kBlk - 1)));
                    }
                    if (!wait_warp(acc_full + slot, (job / C::kSlots) & 1, abort_flag, a.status)) {
                        ok = false;
                    } else {
                        tc_fence_after();
                        float sums[NN];
                        head_sums<NN>(lane_addr + slot * C::kSlotCols, wq, sums, [&] {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(acc_empty + slot);
                        });
#pragma unroll
                        for (int i = 0; i < NN; ++i) {
                            if (s < rs1[i]) {
                                const float v = sums[i] * ksc;
                                a.logits[(static_cast<int64_t>(g) * NN + i) * a.ld + s] = v;
                                if constexpr (TK) {
                                    if (((hb ? hwm1 : hwm0) >> i) & 1u)
                                        atomicAdd(s_hist + (NN * hb + i) * kHistFine + (order_key(v) >> kDigitShift), 1u);
                                }
                            }
                        }
                    }
                }
                ++job;
                if (!ok) {
                    live = false;
                    break;
                }
                new_group = cur.advance(a, s_tiles);
            }
            if constexpr (TK) {
                if (live && have_group) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(hfill + hb);
                    if (flush_pending(true)) {  // the buffer before, then the last group's
                        pend = hb;
                        flush_pending(true);
                    }
                }
            }
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

// -inf for [visible end, ld) of every row.
template <bool P>
__global__ void __launch_bounds__(256) fill_tail_kernel(const LogitsArgs a, int64_t rows) {
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        int64_t start;
        if constexpr (P) {
            const int b = static_cast<int>(r / a.next_n), j = static_cast<int>(r % a.next_n);
            start = decode_row_len(a, __ldg(a.context_lens + b), j, false);
        } else {
            int s0, s1;
            prefill_row_range(a, r, s0, s1, false);
            start = s1 - s0;
        }
        float* row = a.logits + r * a.ld;
        for (int64_t c = start + threadIdx.x; c < a.ld; c += blockDim.x) row[c] = -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[3], s[2];
    cuuint32_t b[3], e[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
    return fn(m, dt, rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool P, int NN, bool TK = false>
int launch(const CUtensorMap& tmK, const CUtensorMap& tmQ,
           const LogitsArgs& a, int64_t rows, int clean, cudaStream_t stream, HistArgs hk = HistArgs{}) {
    hk.group_cost = P ? kGroupCostDecode : kGroupCostPrefill;
    static std::mutex mu;
    static std::vector<char> ready;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IX_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= static_cast<int>(ready.size())) ready.resize(dev + 1, 0);
        if (!ready[dev]) {
            if (cudaFuncSetAttribute(logits_kernel<P, NN, TK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Smem<P, TK>::kAlloc) != cudaSuccess)
                return IX_ERR_CUDA;
            ready[dev] = 1;
        }
    }
    const int sms = num_sms();
    if (sms <= 0) return IX_ERR_CUDA;
    if (a.num_groups > 0) {
        logits_kernel<P, NN, TK><<<sms, kThreads, Smem<P, TK>::kAlloc, stream>>>(tmK, tmQ, a, hk);
        if (launch_status() != IX_OK) return IX_ERR_CUDA;
    }
    if (clean && rows > 0) {
        const int64_t grid = rows < static_cast<int64_t>(sms) * 8 ? rows : static_cast<int64_t>(sms) * 8;
        fill_tail_kernel<P><<<static_cast<int>(grid), 256, 0, stream>>>(a, rows);
        if (launch_status() != IX_OK) return IX_ERR_CUDA;
    }
    return IX_OK;
}

}  // namespace
}  // namespace dsix

using namespace dsix;

namespace dsix {
namespace {

// Host checks of ix_paged_mqa_logits and its fused forms (no CUDA call).
int paged_check(const uint8_t* q_fp8, const float* w, const uint8_t* cache, int64_t num_blocks, int block_size,
                const int32_t* context_lens, const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                int heads, int head_dim, float* logits, int64_t ld, bool* empty) {
    *empty = false;
    if (batch < 0 || num_blocks < 0 || ld < 0 || bt_stride < 0) return IX_ERR_SHAPE;
    if (heads != kHeads || head_dim != kDim || block_size != kBlk || next_n < 1 || next_n > 2)
        return IX_ERR_UNSUPPORTED;
    if (batch == 0 || ld == 0) {
        *empty = true;
        return IX_OK;
    }
    if (ld % 4 != 0 || ld > (1ll << 30)) return IX_ERR_UNSUPPORTED;
    if (num_blocks < 1 || bt_stride < 1) return IX_ERR_SHAPE;
    if (!q_fp8 || !w || !cache || !context_lens || !block_table || !logits) return IX_ERR_NULL;
    if (!aligned16(q_fp8) || !aligned16(w) || !aligned16(cache) || !aligned16(logits))
        return IX_ERR_ALIGN;
    return IX_OK;
}

// Set-up after paged_check: tensor maps and kernel arguments.
int paged_prepare(const uint8_t* q_fp8, const float* w, const uint8_t* cache, int64_t num_blocks,
                  const int32_t* context_lens, const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                  float* logits, int64_t ld, CUtensorMap* tmK, CUtensorMap* tmQ, LogitsArgs* a) {
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    {
        const uint64_t dims[3] = {kDim, kBlk, static_cast<uint64_t>(num_blocks)};
        const uint64_t strides[2] = {kDim, kBlk * (kDim + 4)};
        const uint32_t box[3] = {kDim, kBlk, 1};
        if (!make_map(tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, cache, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return IX_ERR_CUDA;
    }
    {
        const uint64_t dims[2] = {kDim, static_cast<uint64_t>(batch) * next_n * kHeads};
        const uint64_t strides[1] = {kDim};
        const uint32_t box[2] = {kDim, static_cast<uint32_t>(next_n * kHeads)};
        if (!make_map(tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_fp8, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return IX_ERR_CUDA;
    }
    *a = LogitsArgs{};
    a->w = w;
    a->logits = logits;
    a->ld = ld;
    a->num_groups = batch;
    a->status = st;
    a->context_lens = context_lens;
    a->bt = block_table;
    a->bt_stride = bt_stride;
    a->next_n = next_n;
    a->num_blocks = num_blocks;
    a->cache = cache;
    return IX_OK;
}

// Host checks of ix_mqa_logits and its fused forms (no CUDA call).
int contiguous_check(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8, const float* k_scale,
                     const int32_t* ks, const int32_t* ke, int64_t tq, int64_t tk, int heads, int head_dim,
                     float* logits, int64_t ld, bool* empty) {
    *empty = false;
    if (tq < 0 || tk < 0 || ld < 0) return IX_ERR_SHAPE;
    if (heads != kHeads || head_dim != kDim) return IX_ERR_UNSUPPORTED;
    if (tq == 0 || ld == 0) {
        *empty = true;
        return IX_OK;
    }
    if (ld % 4 != 0 || ld > (1ll << 30) || tk >= (1ll << 31) || tq * kHeads >= (1ll << 31))
        return IX_ERR_UNSUPPORTED;
    if (!q_fp8 || !w || !ks || !ke || !logits) return IX_ERR_NULL;
    if (tk > 0 && (!k_fp8 || !k_scale)) return IX_ERR_NULL;
    if (!aligned16(q_fp8) || !aligned16(w) || !aligned16(logits) ||
        (tk > 0 && (!aligned16(k_fp8) || !aligned16(k_scale))))
        return IX_ERR_ALIGN;
    return IX_OK;
}

// Set-up after contiguous_check: tensor maps and kernel arguments.
int contiguous_prepare(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8, const float* k_scale,
                       const int32_t* ks, const int32_t* ke, int64_t tq, int64_t tk, float* logits, int64_t ld,
                       CUtensorMap* tmK, CUtensorMap* tmQ, LogitsArgs* a) {
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    *a = LogitsArgs{};
    a->w = w;
    a->logits = logits;
    a->ld = ld;
    a->num_groups = tk > 0 ? static_cast<int>((tq + Cfg<false>::kRows - 1) / Cfg<false>::kRows) : 0;
    a->status = st;
    a->k_scale = k_scale;
    a->ks = ks;
    a->ke = ke;
    a->tq = tq;
    a->tk = tk;
    *tmK = CUtensorMap{};
    *tmQ = CUtensorMap{};
    if (tk > 0) {
        {
            const uint64_t dims[2] = {kDim, static_cast<uint64_t>(tk)};
            const uint64_t strides[1] = {kDim};
            const uint32_t box[2] = {kDim, kTile};
            if (!make_map(tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, k_fp8, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
                return IX_ERR_CUDA;
        }
        {
            const uint64_t dims[2] = {kDim, static_cast<uint64_t>(tq) * kHeads};
            const uint64_t strides[1] = {kDim};
            const uint32_t box[2] = {kDim, 256};
            if (!make_map(tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_fp8, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
                return IX_ERR_CUDA;
        }
    }
    return IX_OK;
}

// Checks of the histogram arguments (k, workspace) of the *_hist and fused entry points.
int hist_checks(int64_t ld, int k, void* workspace, size_t workspace_bytes, int64_t rows) {
    if (k < 1 || ld > kTopkMaxLd) return IX_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < static_cast<size_t>(rows) * kHistRowWords * 4) return IX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return IX_ERR_ALIGN;
    return IX_OK;
}

}  // namespace
}  // namespace dsix

using namespace dsix;

extern "C" int ix_paged_mqa_logits(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                                   int64_t num_blocks, int block_size,
                                   const int32_t* context_lens, const int32_t* block_table,
                                   int64_t bt_stride, int batch, int next_n, int heads,
                                   int head_dim, float* logits, int64_t ld, int clean_logits,
                                   ix_stream_t stream) {
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = paged_check(q_fp8, w, cache, num_blocks, block_size, context_lens, block_table, bt_stride, batch,
                          next_n, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    chk = paged_prepare(q_fp8, w, cache, num_blocks, context_lens, block_table, bt_stride, batch, next_n, logits,
                        ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    const int64_t rows = static_cast<int64_t>(batch) * next_n;
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    return next_n == 1 ? launch<true, 1>(tmK, tmQ, a, rows, clean_logits, st_)
                       : launch<true, 2>(tmK, tmQ, a, rows, clean_logits, st_);
}

extern "C" int ix_mqa_logits(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                             const float* k_scale, const int32_t* ks, const int32_t* ke, int64_t tq,
                             int64_t tk, int heads, int head_dim, float* logits, int64_t ld,
                             int clean_logits, ix_stream_t stream) {
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = contiguous_check(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    chk = contiguous_prepare(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, logits, ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    return launch<false, 1>(tmK, tmQ, a, tq, clean_logits, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t ix_topk_hist_workspace_size(int64_t rows) {
    return rows > 0 ? static_cast<size_t>(rows) * kHistRowWords * sizeof(uint32_t) : 0;
}

extern "C" int ix_paged_mqa_logits_hist(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                                        int64_t num_blocks, int block_size, const int32_t* context_lens,
                                        const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                                        int heads, int head_dim, float* logits, int64_t ld, int k,
                                        void* workspace, size_t workspace_bytes, ix_stream_t stream) {
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = paged_check(q_fp8, w, cache, num_blocks, block_size, context_lens, block_table, bt_stride, batch,
                          next_n, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    const int64_t rows = static_cast<int64_t>(batch) * next_n;
    chk = hist_checks(ld, k, workspace, workspace_bytes, rows);
    if (chk != IX_OK) return chk;
    chk = paged_prepare(q_fp8, w, cache, num_blocks, context_lens, block_table, bt_stride, batch, next_n, logits,
                        ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    const HistArgs hk{static_cast<uint32_t*>(workspace), k, 0};
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    return next_n == 1 ? launch<true, 1, true>(tmK, tmQ, a, rows, 0, st_, hk) : launch<true, 2, true>(tmK, tmQ, a, rows, 0, st_, hk);
}

extern "C" int ix_mqa_logits_hist(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                                  const float* k_scale, const int32_t* ks, const int32_t* ke, int64_t tq,
                                  int64_t tk, int heads, int head_dim, float* logits, int64_t ld, int k,
                                  void* workspace, size_t workspace_bytes, ix_stream_t stream) {
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = contiguous_check(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    chk = hist_checks(ld, k, workspace, workspace_bytes, tq);
    if (chk != IX_OK) return chk;
    chk = contiguous_prepare(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, logits, ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    const HistArgs hk{static_cast<uint32_t*>(workspace), k, 0};
    return launch<false, 1, true>(tmK, tmQ, a, tq, 0, reinterpret_cast<cudaStream_t>(stream), hk);
}

extern "C" int ix_paged_mqa_logits_topk(const uint8_t* q_fp8, const float* w, const uint8_t* cache,
                                        int64_t num_blocks, int block_size, const int32_t* context_lens,
                                        const int32_t* block_table, int64_t bt_stride, int batch, int next_n,
                                        int heads, int head_dim, float* logits, int64_t ld, int k,
                                        int32_t* out_local, int32_t* out_global, void* workspace,
                                        size_t workspace_bytes, ix_stream_t stream) {
    // every argument is checked before the first launch
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = paged_check(q_fp8, w, cache, num_blocks, block_size, context_lens, block_table, bt_stride, batch,
                          next_n, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    const int64_t rows = static_cast<int64_t>(batch) * next_n;
    chk = hist_checks(ld, k, workspace, workspace_bytes, rows);
    if (chk != IX_OK) return chk;
    if (!out_global) return IX_ERR_NULL;
    chk = paged_prepare(q_fp8, w, cache, num_blocks, context_lens, block_table, bt_stride, batch, next_n, logits,
                        ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    const HistArgs hk{static_cast<uint32_t*>(workspace), k, 0};
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    chk = next_n == 1 ? launch<true, 1, true>(tmK, tmQ, a, rows, 0, st_, hk) : launch<true, 2, true>(tmK, tmQ, a, rows, 0, st_, hk);
    if (chk != IX_OK) return chk;
    SelectRows q{};
    q.logits = logits;
    q.ld = ld;
    q.rows = rows;
    q.context_lens = context_lens;
    q.next_n = next_n;
    q.block_table = block_table;
    q.bt_stride = bt_stride;
    q.block_size = block_size;
    q.k = k;
    q.out_local = out_local;
    q.out_global = out_global;
    q.hist = hk.hist;
    q.status = a.status;
    return select_after_logits(q, st_);
}

extern "C" int ix_mqa_logits_topk(const uint8_t* q_fp8, const float* w, const uint8_t* k_fp8,
                                  const float* k_scale, const int32_t* ks, const int32_t* ke, int64_t tq,
                                  int64_t tk, int heads, int head_dim, float* logits, int64_t ld,
                                  const int32_t* row_req, const int32_t* block_table, int64_t bt_stride,
                                  int block_size, int k, int32_t* out_local, int32_t* out_global,
                                  void* workspace, size_t workspace_bytes, ix_stream_t stream) {
    CUtensorMap tmK, tmQ;
    LogitsArgs a;
    bool empty = false;
    int chk = contiguous_check(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, heads, head_dim, logits, ld, &empty);
    if (chk != IX_OK || empty) return chk;
    chk = hist_checks(ld, k, workspace, workspace_bytes, tq);
    if (chk != IX_OK) return chk;
    if (bt_stride < 0) return IX_ERR_SHAPE;
    if (block_size < 1) return IX_ERR_UNSUPPORTED;
    if (!row_req || !block_table || !out_global) return IX_ERR_NULL;
    chk = contiguous_prepare(q_fp8, w, k_fp8, k_scale, ks, ke, tq, tk, logits, ld, &tmK, &tmQ, &a);
    if (chk != IX_OK) return chk;
    const HistArgs hk{static_cast<uint32_t*>(workspace), k, 0};
    cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    chk = launch<false, 1, true>(tmK, tmQ, a, tq, 0, st_, hk);
    if (chk != IX_OK) return chk;
    SelectRows q{};
    q.logits = logits;
    q.ld = ld;
    q.rows = tq;
    q.ks = ks;
    q.ke = ke;
    q.tk = tk;
    q.row_req = row_req;
    q.block_table = block_table;
    q.bt_stride = bt_stride;
    q.block_size = block_size;
    q.k = k;
    q.out_local = out_local;
    q.out_global = out_global;
    q.hist = hk.hist;
    q.status = a.status;
    return select_after_logits(q, st_);
}
