// topk.cu -- per-row top-k of the indexer logits + remap to global paged-KV slots.
//
// Selection: radix select on an order-preserving 32-bit key of each logit
// (-0.0 folded onto +0.0), up to three digit passes of 11/11/10 bits, then
// one ordered compaction that keeps every key above the threshold and the
// lowest-indexed keys equal to it.  Output is in ascending index order, so
// equal values resolve to the lower index and the result is unique.
//
// GPU layout: a row is split across a thread-block cluster of C CTAs (C = 1,
// 2, 4 or 8, picked on the host from the row length and the row count).  Each
// thread keeps PER consecutive keys of its CTA's slice in registers (read from
// HBM once).  Per pass: shared-memory histogram of the next digit; for C > 1
// the CTAs add their histograms into rank 0's through distributed shared
// memory; one warp of rank 0 finds the digit that holds the k-th largest key
// and writes it into every CTA of the cluster.  Two barriers per pass.  The
// ordered compaction needs one block scan (and, for C > 1, each CTA's count of
// kept keys before its slice, exchanged the same way).  No global scratch.
//
// Short rows (ld <= 16384) with many rows: one WARP per row instead (no block
// barriers; up to 64 rows in flight per SM).  The warp re-reads its row from
// L2 once per pass with coalesced 128-byte loads, counts digits in a
// warp-private shared-memory histogram of packed 16-bit counters, and writes
// the ordered result with ballot/popc positions (coalesced stores).
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsix {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxPer = 64;
constexpr int kSliceCap = kThreads * kMaxPer;  // keys per CTA
constexpr int kBins = 2048;
constexpr int kStage = 4096;  // selected indices staged in shared memory before the write-out
static_assert(kTopkMaxLd == static_cast<int64_t>(kMaxCluster) * kSliceCap, "longest row of the cluster kernel");

struct TopkArgs {
    const float* logits;
    int64_t ld;
    int64_t rows;
    const int32_t* row_len;
    const int32_t* row_req;
    const int32_t* bt;
    int64_t bt_stride;
    int block_size;
    int bs_shift;  // log2(block_size) when it is a power of two, else -1
    int k;
    int32_t* out_local;
    int32_t* out_global;
    int slice;  // keys per CTA (multiple of 4, <= kThreads * PER)
};

enum { kRowsGiven = 0, kRowsDecode = 1, kRowsPrefill = 2 };

// The rows of the selection that follows a histogram logits kernel (a second
// kernel argument, so the plain top-k kernels keep their own).
struct RowsArgs {
    // row geometry: kRowsGiven (row_len / row_req of TopkArgs), kRowsDecode (the
    // paged logits' rows: context_lens, next_n) or kRowsPrefill (ks / ke, tk;
    // row_req), each clamped exactly as the logits kernels clamp them
    int geom;
    const int32_t* context_lens;
    int next_n;
    const int32_t* ks;
    const int32_t* ke;
    int64_t tk;
    // the rows' first-digit histograms written by the logits kernel (read and
    // cleared here); nullptr for the plain top-k
    uint32_t* hist;
    int* status;
};

// Visible length L (clamped to [0, ld]) and request b of row r.
__device__ __forceinline__ void row_geom(const TopkArgs& a, const RowsArgs& f, int64_t r, int64_t& L, int& b) {
    if (f.geom == kRowsDecode) {
        b = static_cast<int>(r / f.next_n);
        L = static_cast<int64_t>(__ldg(f.context_lens + b)) - f.next_n + 1 + r % f.next_n;
    } else if (f.geom == kRowsPrefill) {
        b = __ldg(a.row_req + r);
        int64_t x0 = __ldg(f.ks + r), x1 = __ldg(f.ke + r);
        if (x0 < 0 || x1 > f.tk || x1 < x0) {
            x0 = x0 < 0 ? 0 : x0;
            x1 = x1 > f.tk ? f.tk : x1;
            if (x1 < x0) x1 = x0;
        }
        L = x1 - x0;
    } else {
        b = __ldg(a.row_req + r);
        L = __ldg(a.row_len + r);
    }
    L = L < 0 ? 0 : (L > a.ld ? a.ld : L);
}

__device__ __forceinline__ int warp_incl_scan(int x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// One warp reads the first-digit histogram H of a row with more than k keys
// (64 coarse bins, then 2048 fine bins) and finds the digit d that holds the
// k-th largest key: res = {d, keys in digits above d, keys in d}.  It then
// clears every bin it may have counted (each non-zero coarse bin and its 32
// fine bins), so the workspace is all zero again.  Every lane returns res.
// Returns false when the histogram does not hold exactly the row's L keys (a
// workspace that was not zero before use).
__device__ __forceinline__ bool hist_pick(uint32_t* H, int k, int64_t L, int (&res)[3]) {
    const int lane = threadIdx.x & 31;
    // lane l: coarse bins 63 - 2l (hi) and 62 - 2l (lo); lane 0 holds the top
    const uint2 cc = *reinterpret_cast<const uint2*>(H + 62 - 2 * lane);
    const int c_hi = static_cast<int>(cc.y), c_lo = static_cast<int>(cc.x);
    const int sum = c_hi + c_lo;
    const int incl = warp_incl_scan(sum);
    const bool consistent = __shfl_sync(0xffffffffu, incl, 31) == L;
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= k);
    const int f = hit ? __ffs(hit) - 1 : 31;
    const int excl_f = __shfl_sync(0xffffffffu, incl - sum, f);
    const int chi_f = __shfl_sync(0xffffffffu, c_hi, f);
    const bool in_hi = excl_f + chi_f >= k;
    const int cb = in_hi ? 63 - 2 * f : 62 - 2 * f;
    const int above = in_hi ? excl_f : excl_f + chi_f;
    // the coarse bin's 32 fine bins, lane 0 the highest
    const int fv = static_cast<int>(H[kHistCoarse + cb * 32 + 31 - lane]);
    const int incl2 = warp_incl_scan(fv) + above;
    const unsigned hit2 = __ballot_sync(0xffffffffu, incl2 >= k);
    const int f2 = hit2 ? __ffs(hit2) - 1 : 31;
    res[0] = cb * 32 + 31 - f2;
    res[2] = __shfl_sync(0xffffffffu, fv, f2);
    res[1] = __shfl_sync(0xffffffffu, incl2, f2) - res[2];
    __syncwarp();
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    if (c_hi) {
        uint4* fb = reinterpret_cast<uint4*>(H + kHistCoarse + (63 - 2 * lane) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) fb[i] = z;
    }
    if (c_lo) {
        uint4* fb = reinterpret_cast<uint4*>(H + kHistCoarse + (62 - 2 * lane) * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) fb[i] = z;
    }
    if (sum) *reinterpret_cast<uint2*>(H + 62 - 2 * lane) = make_uint2(0u, 0u);
    return consistent;
}

__device__ __forceinline__ void emit(const TopkArgs& a, int64_t r, int b, int pos, int s) {
    int32_t g = -1;
    if (s >= 0) {
        int q, rem;
        if (a.bs_shift >= 0) {
            q = s >> a.bs_shift;
            rem = s & (a.block_size - 1);
        } else {
            q = s / a.block_size;
            rem = s % a.block_size;
        }
        const int64_t blk = __ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + q);
        g = static_cast<int32_t>(blk * a.block_size + rem);
    }
    if (a.out_local) a.out_local[r * a.k + pos] = s;
    a.out_global[r * a.k + pos] = g;
}

// Block-wide exclusive scan of a uint32 per thread (wrapping adds); *total = sum.
__device__ __forceinline__ uint32_t scan_excl(uint32_t v, uint32_t* scratch, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const uint32_t s = lane < kWarps ? scratch[lane] : 0u;
        uint32_t inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < kWarps) scratch[32 + lane] = inc - s;
        if (lane == kWarps - 1) scratch[64] = inc;
    }
    __syncthreads();
    const uint32_t r = scratch[32 + warp] + x - v;
    *total = scratch[64];
    return r;
}

// Block-wide digit pick over histogram h of nb bins (a power of two <= 2048):
// thread t owns max(nb / kThreads, 1) consecutive bins counted from the top
// (thread 0 the highest), zeroes them after reading, and the thread whose
// range holds the k_rem-th key writes {digit, keys above it, keys in it} to out.
// Ends with a barrier.
__device__ __forceinline__ void block_pick(int* h, int nb, int k_rem, int* out, uint32_t* scratch) {
    constexpr int kMaxPer = kBins / kThreads;
    const int tid = threadIdx.x;
    const int per = nb >= kThreads ? nb / kThreads : 1;
    const int base = nb - per * (tid + 1);  // negative: no bin for this thread (nb < kThreads)
    int c[kMaxPer];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        c[i] = (i < per && base + i >= 0) ? h[base + i] : 0;
        sum += c[i];
    }
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i)
        if (i < per && base + i >= 0) h[base + i] = 0;
    uint32_t tot;
    const int above = static_cast<int>(scan_excl(static_cast<uint32_t>(sum), scratch, &tot));
    if (above < k_rem && above + sum >= k_rem) {
        int acc = above;
#pragma unroll
        for (int i = kMaxPer - 1; i >= 0; --i) {
            if (i < per && base + i >= 0 && acc + c[i] >= k_rem) {
                out[0] = base + i;
                out[1] = acc;
                out[2] = c[i];
                break;
            }
            acc += c[i];
        }
    }
    __syncthreads();
}

// Short slices keep several CTAs per SM resident to hide the per-row phase latency.
// HIST: the rows' first-digit histograms come from the logits kernel, so the
// key min / max and the first histogram pass over all keys are skipped.
template <int PER, bool HIST>
__global__ void __launch_bounds__(kThreads, PER <= 4 ? 3 : (PER <= 32 ? 2 : 1))
    topk_kernel(const TopkArgs a, const RowsArgs f) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, warp = tid >> 5;

    __shared__ int hist[kBins];
    __shared__ int merged[kBins];            // rank 0 only, for C > 1
    __shared__ int counts[2 * kMaxCluster];  // rank 0 only
    __shared__ int res[4];                   // digit, count above, count in bin
    __shared__ uint32_t scratch[72];
    __shared__ int stage[kStage];            // this CTA's kept indices, in output order
    __shared__ uint32_t mmx[2 * (kThreads / 32)];  // per-warp key min / max
    __shared__ uint32_t cmm[2 * kMaxCluster];      // per-CTA key min / max (rank 0's copy is read)

    for (int i = tid; i < kBins; i += kThreads) {
        hist[i] = 0;
        merged[i] = 0;
    }
    cluster.sync();
    int* merged0 = cluster.map_shared_rank(merged, 0);
    int* counts0 = cluster.map_shared_rank(counts, 0);
    uint32_t* cmm0 = cluster.map_shared_rank(cmm, 0);

    const int64_t cid = blockIdx.x / C;
    const int64_t nclusters = gridDim.x / C;
    for (int64_t r = cid; r < a.rows; r += nclusters) {
        int64_t L;
        int b;
        row_geom(a, f, r, L, b);
        if (L <= a.k) {
            for (int i = rank * kThreads + tid; i < a.k; i += C * kThreads)
                emit(a, r, b, i, i < L ? i : -1);
            continue;  // uniform over the cluster
        }
        const int lo = rank * a.slice;
        const int64_t avail = L - lo;
        const int n = avail <= 0 ? 0 : static_cast<int>(avail < a.slice ? avail : a.slice);
        const int mine = tid * PER;                        // first slice index of this thread
        const int nv = max(0, min(PER, n - mine));         // valid keys of this thread
        const float* src = a.logits + r * a.ld + lo + mine;  // 16-byte aligned
        uint32_t key[PER];
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
        for (int j = 0; j < PER; j += 4) {
            if (j + 4 <= nv) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(src + j));
                key[j] = order_key(v.x);
                key[j + 1] = order_key(v.y);
                key[j + 2] = order_key(v.z);
                key[j + 3] = order_key(v.w);
                kmin = min(kmin, min(min(key[j], key[j + 1]), min(key[j + 2], key[j + 3])));
                kmax = max(kmax, max(max(key[j], key[j + 1]), max(key[j + 2], key[j + 3])));
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    key[j + q] = 0u;
                    if (j + q < nv) {
                        key[j + q] = order_key(__ldg(src + j + q));
                        kmin = min(kmin, key[j + q]);
                        kmax = max(kmax, key[j + q]);
                    }
                }
            }
        }
        int shift, k_rem;
        uint32_t prefix;
        bool done;
        if constexpr (HIST) {
            // the threshold digit from the row's histogram: one warp of rank 0
            // reads (and clears) it and hands the result to every CTA
            if (rank == 0 && warp == 0) {
                int hr[3];
                if (!hist_pick(f.hist + r * kHistRowWords, a.k, L, hr) && tid == 0) flag(f.status, IX_DEV_BAD_HIST);
                if ((tid & 31) < 3)
                    for (int j = 0; j < C; ++j) cluster.map_shared_rank(res, j)[tid & 31] = hr[tid & 31];
            }
            if (C > 1)
                cluster.sync();
            else
                __syncthreads();
            shift = kDigitShift;
            prefix = static_cast<uint32_t>(res[0]);
            k_rem = a.k - res[1];
            done = res[2] == k_rem;
        } else {
            // Bits every key of the row shares need no histogram (a row of logits
            // often spans one or two binades): the digits start below them.  Key
            // min / max over the row: warps, then CTAs through rank 0.
            kmin = __reduce_min_sync(0xffffffffu, kmin);
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            if ((tid & 31) == 0) {
                mmx[2 * warp] = kmin;
                mmx[2 * warp + 1] = kmax;
            }
            __syncthreads();
            if (tid == 0) {
                for (int i = 1; i < kThreads / 32; ++i) {
                    kmin = min(kmin, mmx[2 * i]);
                    kmax = max(kmax, mmx[2 * i + 1]);
                }
                cmm0[2 * rank] = kmin;
                cmm0[2 * rank + 1] = kmax;
            }
            if (C > 1)
                cluster.sync();
            else
                __syncthreads();
            kmin = cmm0[0];
            kmax = cmm0[1];
#pragma unroll
            for (int i = 1; i < kMaxCluster; ++i) {  // unrolled: the remote loads go out together
                if (i < C) {
                    kmin = min(kmin, cmm0[2 * i]);
                    kmax = max(kmax, cmm0[2 * i + 1]);
                }
            }
            shift = 32 - __clz(kmin ^ kmax);  // bits below the common prefix; 0 when all keys are equal
            prefix = shift >= 32 ? 0u : (kmin >> shift);
            k_rem = a.k;
            done = shift == 0;
        }
        for (int p = 0; !done; ++p) {
            const int nbits = shift < 11 ? shift : 11;
            const int nb = 1 << nbits;
            const int sh = shift - nbits;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                if (j < nv && ((!HIST && p == 0) || (key[j] >> shift) == prefix))
                    atomicAdd(hist + ((key[j] >> sh) & (nb - 1)), 1);
            }
            if (C > 1) {
                cluster.sync();  // every CTA's histogram of this pass is complete
                // distributed merge: each bin is summed by one thread of the cluster
                for (int i = rank * kThreads + tid; i < nb; i += C * kThreads) {
                    int sum = 0;
                    for (int j = 0; j < C; ++j) sum += cluster.map_shared_rank(hist, j)[i];
                    merged0[i] = sum;
                }
                cluster.sync();  // merged bins complete; no CTA reads another's histogram now
                for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
                if (rank == 0) {
                    block_pick(merged, nb, k_rem, res, scratch);
                    if (tid < 3)
                        for (int j = 1; j < C; ++j) cluster.map_shared_rank(res, j)[tid] = res[tid];
                }
                cluster.sync();
            } else {
                __syncthreads();
                block_pick(hist, nb, k_rem, res, scratch);
            }
            k_rem -= res[1];
            prefix = (shift >= 32 ? 0u : (prefix << nbits)) | static_cast<uint32_t>(res[0]);
            shift = sh;
            done = shift == 0 || res[2] == k_rem;  // every key of this digit is kept
        }
        // kept: keys with (u >> shift) > prefix, and the first k_rem equal to it
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            if (j < nv) {
                const uint32_t v = key[j] >> shift;
                gt += v > prefix;
                eq += v == prefix;
            }
        }
        uint32_t tot;
        const uint32_t ex = scan_excl((gt << 16) | eq, scratch, &tot);  // fields < 2^16 per CTA
        int bg = static_cast<int>(ex >> 16), be = static_cast<int>(ex & 0xFFFFu);
        int carry_gt = 0, carry_eq = 0;
        if (C > 1) {
            if (tid == 0) {
                counts0[2 * rank] = static_cast<int>(tot >> 16);
                counts0[2 * rank + 1] = static_cast<int>(tot & 0xFFFFu);
            }
            cluster.sync();
            for (int j = 0; j < rank; ++j) {
                carry_gt += counts0[2 * j];
                carry_eq += counts0[2 * j + 1];
            }
            bg += carry_gt;
            be += carry_eq;
        }
        // this CTA's kept keys occupy output positions [cstart, cend)
        const int cstart = carry_gt + min(carry_eq, k_rem);
        const int cend = min(a.k, carry_gt + static_cast<int>(tot >> 16) +
                                      min(carry_eq + static_cast<int>(tot & 0xFFFFu), k_rem));
        const bool staged = cstart >= 0 && cend - cstart <= kStage;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            if (j < nv) {
                const uint32_t v = key[j] >> shift;
                const bool g = v > prefix, e = v == prefix;
                const int pos = bg + min(be, k_rem);
                if ((g || (e && be < k_rem)) && pos >= 0 && pos < a.k) {
                    if (staged) {
                        if (pos >= cstart && pos - cstart < kStage) stage[pos - cstart] = lo + mine + j;
                    } else {
                        emit(a, r, b, pos, lo + mine + j);
                    }
                }
                bg += g;
                be += e;
            }
        }
        if (staged) {  // coalesced write-out with the remap
            __syncthreads();
            for (int i = tid; i < cend - cstart; i += kThreads) emit(a, r, b, cstart + i, stage[i]);  // cstart >= 0, cend <= k
        }
        // res, scratch and counts are rewritten only after barriers that every
        // thread of the cluster reaches after its reads above
        __syncthreads();
    }
    cluster.sync();  // no CTA leaves while another may still touch its shared memory
}


// ---------------------------------------------------------------------------
// Short rows (ld <= 16384, many rows): one 256-thread CTA per row, no cluster.
// Keys live in registers (PER consecutive keys per thread), so the row crosses
// HBM once; each pass is a shared-memory histogram, then a block-wide digit
// pick (up to 8 bins per thread, one block scan).  The request's block-table
// row is staged in shared memory for the remap.
// ---------------------------------------------------------------------------
constexpr int kBlkThreads = 256;
constexpr int kBlkWarps = kBlkThreads / 32;
constexpr int kBlkMaxLd = 16384;
constexpr int kBlkBt = 256;  // block-table entries staged (16384 keys at block size 64), one per thread
static_assert(kBlkBt == kBlkThreads, "one staged block-table entry per thread");
constexpr int kBlkBits = 12;  // radix digit width: 12 + 12 + 8 bits cover a 32-bit key
constexpr int kBlkBins = 1 << kBlkBits;
constexpr int kBlkFewKeys = 1024;  // threshold-bin size below which later passes take 10-bit digits
constexpr int kBlkRankKeys = 128;  // threshold-bin size up to which its keys are ranked directly

__device__ __forceinline__ uint32_t blk_scan_excl(uint32_t v, uint32_t* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int i = 0; i < kBlkWarps; ++i) before += i < warp ? scratch[i] : 0u;
    return before + x - v;
}

constexpr int kBlkStage = 2048;  // largest k whose winners are staged in shared memory

// Remap of local key index s (< row length) through the request's block-table
// row, read from shared memory when it was staged there.
// btrow holds the staged entries already multiplied by the block size (low 32
// bits, the same value the int64 product is narrowed to).
__device__ __forceinline__ int32_t remap_row(const TopkArgs& a, const int32_t* btrow, bool bt_staged, int b, int s) {
    if (bt_staged && a.bs_shift >= 0) return btrow[s >> a.bs_shift] + (s & (a.block_size - 1));
    const int64_t blk = __ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + s / a.block_size);
    return static_cast<int32_t>(blk * a.block_size + s % a.block_size);
}

template <int PER>
struct BlkMask;  // one bit per key slot of a thread
template <>
struct BlkMask<32> {
    using T = uint32_t;
};
template <>
struct BlkMask<64> {
    using T = unsigned long long;
};
__device__ __forceinline__ int mask_popc(uint32_t m) { return __popc(m); }
__device__ __forceinline__ int mask_popc(unsigned long long m) { return __popcll(m); }
__device__ __forceinline__ int mask_low(uint32_t m) { return __ffs(m) - 1; }
__device__ __forceinline__ int mask_low(unsigned long long m) { return __ffsll(m) - 1; }

// Slots past the row end hold key 0 and stay out of every histogram.  Key 0 is
// below the key of every finite value and those slots come after every real
// key in index order, so even when the threshold bin starts at 0 they are past
// the k_rem equal keys that are taken.
template <int PER>
__global__ void __launch_bounds__(kBlkThreads, PER <= 32 ? 4 : 2) topk_block_kernel(const TopkArgs a) {
    using mask_t = typename BlkMask<PER>::T;
    __shared__ __align__(16) int hist[kBlkBins];
    __shared__ int32_t btrow[kBlkBt];
    __shared__ uint32_t scratch[2][kBlkWarps];
    __shared__ uint32_t mm[2][kBlkWarps];
    __shared__ int res[4];
    __shared__ uint32_t taken[kBlkWarps];  // ranked bin: bit i of word w = candidate 32 w + i is taken
    __shared__ __align__(16) int32_t stage[kBlkStage];
    const int tid = threadIdx.x;
    for (int i = tid; i < kBlkBins; i += kBlkThreads) hist[i] = 0;
    __syncthreads();
    int sc = 0;  // alternates the scan scratch so back-to-back scans need no extra barrier
    // A row's length and request are read one row ahead, and its block-table
    // entries are loaded before the row and stored to shared memory only after
    // the first barrier, so no global load waits on another at the row start.
    int64_t len_nx = blockIdx.x < a.rows ? __ldg(a.row_len + blockIdx.x) : 0;
    int req_nx = blockIdx.x < a.rows ? __ldg(a.row_req + blockIdx.x) : 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        int64_t L64 = len_nx;
        L64 = L64 < 0 ? 0 : (L64 > a.ld ? a.ld : L64);
        const int L = static_cast<int>(L64);
        const int b = req_nx;
        if (r + gridDim.x < a.rows) {
            len_nx = __ldg(a.row_len + r + gridDim.x);
            req_nx = __ldg(a.row_req + r + gridDim.x);
        }
        if (L <= a.k) {
            for (int i = tid; i < a.k; i += kBlkThreads) emit(a, r, b, i, i < L ? i : -1);
            continue;
        }
        const int nblk = (L + a.block_size - 1) / a.block_size;
        const bool bt_staged = nblk <= kBlkBt;  // kBlkBt == kBlkThreads: one entry per thread
        const bool bt_mine = bt_staged && a.bs_shift >= 0 && tid < nblk;
        uint32_t btv = 0;
        if (bt_mine) btv = static_cast<uint32_t>(__ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + tid));
        const int mine = tid * PER;
        const int nv = max(0, min(PER, L - mine));
        const float* src = a.logits + r * a.ld + mine;  // 16-byte aligned
        uint32_t key[PER];
        uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
        // Threads past the row end (whole warps of a short row) skip every loop
        // over their key slots; their slots hold 0 and count nowhere.
        if (nv > 0) {
#pragma unroll
            for (int j = 0; j < PER; j += 4) {
                if (j + 4 <= nv) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(src + j));
                    key[j] = order_key(v.x);
                    key[j + 1] = order_key(v.y);
                    key[j + 2] = order_key(v.z);
                    key[j + 3] = order_key(v.w);
                    kmin = min(kmin, min(min(key[j], key[j + 1]), min(key[j + 2], key[j + 3])));
                    kmax = max(kmax, max(max(key[j], key[j + 1]), max(key[j + 2], key[j + 3])));
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        key[j + q] = 0u;
                        if (j + q < nv) {
                            key[j + q] = order_key(__ldg(src + j + q));
                            kmin = min(kmin, key[j + q]);
                            kmax = max(kmax, key[j + q]);
                        }
                    }
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) key[j] = 0u;
        }
        // Bits every key of the row shares need no histogram.  A row of logits
        // often spans one or two binades, so a first digit taken from the sign
        // and exponent would send nearly every key to a few bins and serialise
        // the shared-memory atomics; the digits start below the common prefix.
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if ((tid & 31) == 0) {
            mm[0][tid >> 5] = kmin;
            mm[1][tid >> 5] = kmax;
        }
        __syncthreads();
        if (bt_mine) btrow[tid] = static_cast<int32_t>(btv * static_cast<uint32_t>(a.block_size));
#pragma unroll
        for (int i = 0; i < kBlkWarps; ++i) {
            kmin = min(kmin, mm[0][i]);
            kmax = max(kmax, mm[1][i]);
        }
        int shift = 32 - __clz(kmin ^ kmax);  // bits below the common prefix; 0 when all keys are equal
        uint32_t prefix = shift >= 32 ? 0u : (kmin >> shift);
        int k_rem = a.k;
        bool done = shift == 0, ranked = false;
        for (int p = 0; !done; ++p) {
            // after the first pass few keys remain in the threshold bin: a 10-bit
            // digit (four bins per thread in the pick) usually settles them
            const int width = (p > 0 && res[2] <= kBlkFewKeys) ? 10 : kBlkBits;
            const int nbits = shift < width ? shift : width;
            const int nb = 1 << nbits;
            const int sh = shift - nbits;
            if (nv == 0) {
            } else if (p == 0) {
#pragma unroll
                for (int j = 0; j < PER; j += 4) {
                    if (j + 4 <= nv) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) atomicAdd(hist + ((key[j + q] >> sh) & (nb - 1)), 1);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (j + q < nv) atomicAdd(hist + ((key[j + q] >> sh) & (nb - 1)), 1);
                    }
                }
            } else {
                // few keys are left in the bin: one predicated atomic per key in it
#pragma unroll
                for (int j = 0; j < PER; ++j)
                    if (j < nv && (key[j] >> shift) == prefix) atomicAdd(hist + ((key[j] >> sh) & (nb - 1)), 1);
            }
            __syncthreads();
            // Block-wide pick: thread t owns max(nb / 256, 1) consecutive bins
            // counted from the top (thread 0 the highest; with fewer than 256
            // bins the threads past nb own none).  Owners read their bins with
            // 16-byte loads; the thread whose range holds the k_rem-th key walks
            // its bins again, and every owner clears its bins before the barrier
            // that publishes the digit.
            const int per = nb >= kBlkThreads ? nb / kBlkThreads : 1;
            const int base = nb - per * (tid + 1);
            int sum = 0;
            if (per >= 4) {
                const int4* h4 = reinterpret_cast<const int4*>(hist + base);  // base is a multiple of 4
                for (int i = 0; i < per / 4; ++i) {
                    const int4 v = h4[i];
                    sum += (v.x + v.y) + (v.z + v.w);
                }
            } else if (base >= 0) {
                for (int i = 0; i < per; ++i) sum += hist[base + i];
            }
            const int above = static_cast<int>(blk_scan_excl(static_cast<uint32_t>(sum), scratch[sc]));
            sc ^= 1;
            if (above < k_rem && above + sum >= k_rem) {
                int acc = above;
                if (per >= 4) {  // 16-byte steps from the top bin down
                    const int4* h4 = reinterpret_cast<const int4*>(hist + base);
                    for (int i = per / 4 - 1; i >= 0; --i) {
                        const int4 v = h4[i];
                        bool found = false;
                        int bin = 0, cnt_bin = 0, acc_bin = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // bins base + 4i + 3 down to base + 4i
                            const int cnt = q == 0 ? v.w : (q == 1 ? v.z : (q == 2 ? v.y : v.x));
                            if (!found) {
                                if (acc + cnt >= k_rem) {
                                    found = true;
                                    bin = base + 4 * i + 3 - q;
                                    cnt_bin = cnt;
                                    acc_bin = acc;
                                } else {
                                    acc += cnt;
                                }
                            }
                        }
                        if (found) {
                            res[0] = bin;
                            res[1] = acc_bin;
                            res[2] = cnt_bin;
                            break;
                        }
                    }
                } else {
                    for (int i = per - 1; i >= 0; --i) {
                        const int cnt = hist[base + i];
                        if (acc + cnt >= k_rem) {
                            res[0] = base + i;
                            res[1] = acc;
                            res[2] = cnt;
                            break;
                        }
                        acc += cnt;
                    }
                }
            }
            if (per >= 4) {
                int4* h4 = reinterpret_cast<int4*>(hist + base);
                for (int i = 0; i < per / 4; ++i) h4[i] = make_int4(0, 0, 0, 0);
            } else if (base >= 0) {
                for (int i = 0; i < per; ++i) hist[base + i] = 0;
            }
            __syncthreads();
            k_rem -= res[1];
            prefix = (shift >= 32 ? 0u : (prefix << nbits)) | static_cast<uint32_t>(res[0]);
            shift = sh;
            done = shift == 0 || res[2] == k_rem;
            if (!done && res[2] <= kBlkRankKeys) {  // few keys left in the bin: rank them below
                done = true;
                ranked = true;
            }
        }
        // Keys above the threshold bin are all taken; of the keys in it, the
        // first k_rem in index order (all of them when the bin holds exactly k_rem).
        const uint32_t thr_lo = prefix << shift;
        const uint32_t thr_hi = thr_lo | ((1u << shift) - 1u);
        mask_t gm = 0, em = 0;
        if (nv > 0) {
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                gm |= key[j] > thr_hi ? (mask_t(1) << j) : mask_t(0);
                em |= key[j] >= thr_lo ? (mask_t(1) << j) : mask_t(0);
            }
            em &= ~gm;
        }
        const int pg = mask_popc(gm), pe = mask_popc(em);
        const uint32_t ex = blk_scan_excl((static_cast<uint32_t>(pg) << 16) | static_cast<uint32_t>(pe),
                                          scratch[sc]);  // both fields stay below 2^16
        sc ^= 1;
        const int bg = static_cast<int>(ex >> 16), be = static_cast<int>(ex & 0xFFFFu);
        mask_t sel = gm;
        int pos;
        if (ranked) {
            // The bin's n <= kBlkRankKeys keys, numbered in index order (this
            // thread's are be .., its keys re-read from L1/L2), go to shared
            // memory; candidate i is taken when fewer than k_rem candidates
            // rank above it (a larger key, or an equal key at a lower index).
            const int n = res[2];
            uint32_t* cand = reinterpret_cast<uint32_t*>(stage);  // stage is written only after the next barrier
            // only keys before the row end count (a bin at key 0 would also hold the
            // padding slots), and no index leaves [0, n)
            em &= nv >= PER ? ~mask_t(0) : ((mask_t(1) << nv) - 1);
            const int b0 = min(be, n);
            {
                mask_t e = em;
                int c = b0;
                while (e && c < n) {
                    cand[c++] = order_key(__ldg(src + mask_low(e)));
                    e &= e - 1;
                }
            }
            __syncthreads();
            bool tk = false;
            if (tid < n) {
                const uint32_t kt = cand[tid];
                int above = 0;
                for (int u = 0; u < n; ++u) {
                    const uint32_t ku = cand[u];
                    above += (ku > kt || (ku == kt && u < tid)) ? 1 : 0;
                }
                tk = above < k_rem;
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, tk);
            if ((tid & 31) == 0) taken[tid >> 5] = bal;
            __syncthreads();
            // this thread's candidates be .. be + pe - 1, and the taken ones before them
            int before = 0;
            for (int w = 0; w < (b0 >> 5); ++w) before += __popc(taken[w]);
            if (b0 & 31) before += __popc(taken[b0 >> 5] & ((1u << (b0 & 31)) - 1u));
            mask_t e = em;
            int c = b0;
            while (e && c < n) {
                const mask_t low = e & (~e + 1);
                if ((taken[c >> 5] >> (c & 31)) & 1u) sel |= low;
                ++c;
                e &= e - 1;
            }
            pos = bg + before;
        } else {
            const int take = max(0, min(pe, k_rem - be));
            if (take == pe) {
                sel |= em;
            } else if (take > 0) {
                mask_t rest = em;
                for (int i = 0; i < take; ++i) rest &= rest - 1;
                sel |= em ^ rest;
            }
            pos = bg + min(be, k_rem);
        }
        // The winners of one thread are consecutive positions, so lanes write
        // far-apart runs; for k <= kBlkStage the local indices are placed in
        // shared memory first and both outputs leave in coalesced order, with the
        // remap done only for the k winners.
        const bool staged = a.k <= kBlkStage;
        int32_t* __restrict__ og = a.out_global + r * a.k;
        int32_t* __restrict__ ol = a.out_local ? a.out_local + r * a.k : nullptr;
        while (sel) {
            const int s = mine + mask_low(sel);
            sel &= sel - 1;
            if (pos >= 0 && pos < a.k) {
                if (staged) {
                    stage[pos] = s;
                } else {
                    og[pos] = remap_row(a, btrow, bt_staged, b, s);
                    if (ol) ol[pos] = s;
                }
            }
            ++pos;
        }
        if (staged) {
            __syncthreads();
            // four outputs per thread and step, 16-byte stores when the rows allow
            const bool vec = (a.k & 3) == 0 &&
                             ((reinterpret_cast<uintptr_t>(a.out_global) |
                               reinterpret_cast<uintptr_t>(a.out_local)) & 15u) == 0;
            if (vec) {
                for (int i = 4 * tid; i < a.k; i += 4 * kBlkThreads) {
                    const int4 s4 = *reinterpret_cast<const int4*>(stage + i);
                    *reinterpret_cast<int4*>(og + i) =
                        make_int4(remap_row(a, btrow, bt_staged, b, s4.x), remap_row(a, btrow, bt_staged, b, s4.y),
                                  remap_row(a, btrow, bt_staged, b, s4.z), remap_row(a, btrow, bt_staged, b, s4.w));
                    if (ol) *reinterpret_cast<int4*>(ol + i) = s4;
                }
            } else {
                for (int i = tid; i < a.k; i += kBlkThreads) {
                    const int s = stage[i];
                    og[i] = remap_row(a, btrow, bt_staged, b, s);
                    if (ol) ol[i] = s;
                }
            }
        }
        __syncthreads();  // btrow, mm, res and stage are rewritten by the next row
    }
}

// ---------------------------------------------------------------------------
// Fused path, many rows: one WARP per row, finishing the selection that the
// logits kernel started with the row's first-digit histogram.  No block
// barriers, up to 48 rows in flight per SM.
//   1. hist_pick: the digit d that holds the k-th largest key, the keys above
//      it (all selected) and the count c of keys in it.
//   2. If not all c keys of d are taken: the keys of digit d (read from the
//      logits row once) go to shared memory when c <= kSelCap,
//      and 7-bit radix levels over them settle the remaining 21 bits; past
//      kSelCap the levels re-read the row instead.  The result is a prefix of
//      the key (of `sh` bits below the top) above which everything is taken,
//      and `take`: how many keys equal to the prefix are taken, the lowest
//      indices first.
//   3. One pass over the row emits the selection in ascending index order
//      with the remap (ballot/popc positions, stores in order).
// ---------------------------------------------------------------------------
constexpr int kSelWarps = 8;
constexpr int kSelCap = 512;
constexpr int kSelBits = 7;

// Warp-wide pick over `nb` (<= 128) bins h[] from the top: lane l owns bins
// nb-1-4l .. nb-4-4l.  Returns the bin holding the take-th key, the keys above
// it and the keys in it (every lane).
__device__ __forceinline__ void warp_pick(const uint32_t* h, int nb, int take, int& d, int& above, int& cnt) {
    const int lane = threadIdx.x & 31;
    int c[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int bin = nb - 1 - 4 * lane - q;
        c[q] = bin >= 0 ? static_cast<int>(h[bin]) : 0;
        sum += c[q];
    }
    const int incl = warp_incl_scan(sum);
    const unsigned hit = __ballot_sync(0xffffffffu, incl >= take);
    const int f = hit ? __ffs(hit) - 1 : 31;
    int dd = 0, ab = 0, cn = 0;
    if (lane == f) {
        int acc = incl - sum;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (acc + c[q] >= take || q == 3) {
                dd = nb - 1 - 4 * lane - q;
                ab = acc;
                cn = c[q];
                break;
            }
            acc += c[q];
        }
    }
    d = __shfl_sync(0xffffffffu, dd, f);
    above = __shfl_sync(0xffffffffu, ab, f);
    cnt = __shfl_sync(0xffffffffu, cn, f);
}

// Keys of the 128-key chunk starting at c0 held by this lane (keys c0 + 4 lane
// .. + 3); valid bits for keys below L.
__device__ __forceinline__ unsigned chunk_keys(const float* row, int c0, int L, uint32_t (&key)[4]) {
    const int i0 = c0 + 4 * (threadIdx.x & 31);
    unsigned valid = 0;
    if (i0 < L) {  // i0 + 3 < ld: ld is a multiple of 4 and L <= ld
        const float4 v = __ldg(reinterpret_cast<const float4*>(row + i0));
        key[0] = order_key(v.x);
        key[1] = order_key(v.y);
        key[2] = order_key(v.z);
        key[3] = order_key(v.w);
        const int n = L - i0;
        valid = n >= 4 ? 0xFu : ((1u << n) - 1u);
    } else {
        key[0] = key[1] = key[2] = key[3] = 0u;
    }
    return valid;
}

__device__ __forceinline__ int warp_excl_scan(int x, int& total) {
    const int incl = warp_incl_scan(x);
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - x;
}

__global__ void __launch_bounds__(kSelWarps * 32) select_warp_kernel(const TopkArgs a, const RowsArgs f) {
    __shared__ uint32_t s_key[kSelWarps][kSelCap];
    __shared__ uint32_t s_h[kSelWarps][1 << kSelBits];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t* ck = s_key[warp];
    uint32_t* wh = s_h[warp];
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kSelWarps;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kSelWarps + warp; r < a.rows; r += nw) {
        int64_t L64;
        int b;
        row_geom(a, f, r, L64, b);
        const int L = static_cast<int>(L64);
        if (L <= a.k) {
            for (int i = lane; i < a.k; i += 32) emit(a, r, b, i, i < L ? i : -1);
            continue;
        }
        int hr[3];
        if (!hist_pick(f.hist + r * kHistRowWords, a.k, L, hr) && lane == 0) flag(f.status, IX_DEV_BAD_HIST);
        uint32_t prefix = static_cast<uint32_t>(hr[0]);
        int take = a.k - hr[1], cnt = hr[2], sh = kDigitShift;
        const float* row = a.logits + r * a.ld;
        if (cnt != take) {
            const bool in_smem = cnt <= kSelCap;
            int ncand = 0;
            if (in_smem) {  // the keys of the threshold digit, in index order
                for (int c0 = 0; c0 < L; c0 += 128) {
                    uint32_t key[4];
                    const unsigned valid = chunk_keys(row, c0, L, key);
                    unsigned eq = 0;
#pragma unroll
                    for (int j = 0; j < 4; ++j) eq |= (((valid >> j) & 1u) && (key[j] >> sh) == prefix) ? (1u << j) : 0u;
                    int tot;
                    int pos = ncand + warp_excl_scan(__popc(eq), tot);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if ((eq >> j) & 1u) {
                            if (pos < kSelCap) ck[pos] = key[j];
                            ++pos;
                        }
                    }
                    ncand += tot;
                }
                ncand = min(ncand, kSelCap);
                __syncwarp();
            }
            while (cnt != take && sh > 0) {
                const int nb = sh < kSelBits ? sh : kSelBits, nsh = sh - nb;
                const uint32_t m = (1u << nb) - 1u;
                for (int i = lane; i < (1 << kSelBits); i += 32) wh[i] = 0u;
                __syncwarp();
                if (in_smem) {
                    for (int i = lane; i < ncand; i += 32) {
                        const uint32_t key = ck[i];
                        if ((key >> sh) == prefix) atomicAdd(wh + ((key >> nsh) & m), 1u);
                    }
                } else {
                    for (int c0 = 0; c0 < L; c0 += 128) {
                        uint32_t key[4];
                        const unsigned valid = chunk_keys(row, c0, L, key);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (((valid >> j) & 1u) && (key[j] >> sh) == prefix) atomicAdd(wh + ((key[j] >> nsh) & m), 1u);
                    }
                }
                __syncwarp();
                int d, above, c;
                warp_pick(wh, 1 << nb, take, d, above, c);
                prefix = (prefix << nb) | static_cast<uint32_t>(d);
                take -= above;
                cnt = c;
                sh = nsh;
                __syncwarp();
            }
        }
        // emit: keys above the prefix, and the first `take` keys equal to it
        int pos0 = 0, eq0 = 0;
        for (int c0 = 0; c0 < L; c0 += 128) {
            uint32_t key[4];
            const unsigned valid = chunk_keys(row, c0, L, key);
            unsigned gt = 0, eq = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if ((valid >> j) & 1u) {
                    const uint32_t v = key[j] >> sh;
                    gt |= v > prefix ? (1u << j) : 0u;
                    eq |= v == prefix ? (1u << j) : 0u;
                }
            }
            int eq_tot;
            int er = eq0 + warp_excl_scan(__popc(eq), eq_tot);
            unsigned sel = gt;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if ((eq >> j) & 1u) {
                    if (er < take) sel |= 1u << j;
                    ++er;
                }
            }
            int s_tot;
            int pos = pos0 + warp_excl_scan(__popc(sel), s_tot);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if ((sel >> j) & 1u) {
                    if (pos < a.k) emit(a, r, b, pos, c0 + 4 * lane + j);
                    ++pos;
                }
            }
            pos0 += s_tot;
            eq0 += eq_tot;
        }
        if (pos0 != a.k) {  // the histogram did not match the row: workspace not cleared before use
            if (lane == 0) flag(f.status, IX_DEV_BAD_HIST);
            for (int i = pos0 + lane; i < a.k; i += 32) emit(a, r, b, i, -1);
        }
    }
}

template <int PER, bool HIST>
int cluster_setup() {  // the carve-out attribute, once per device
    static std::mutex mu;
    static std::vector<char> ready;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(ready.size())) ready.resize(dev + 1, 0);
    if (!ready[dev]) {
        if (cudaFuncSetAttribute(topk_kernel<PER, HIST>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return IX_ERR_CUDA;
        ready[dev] = 1;
    }
    return IX_OK;
}

template <int PER, bool HIST>
int launch_per(const TopkArgs& a, const RowsArgs& f, int C, int64_t clusters, cudaStream_t stream) {
    const int st = cluster_setup<PER, HIST>();
    if (st != IX_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk_kernel<PER, HIST>, a, f) != cudaSuccess) {
        cudaGetLastError();
        return IX_ERR_CUDA;
    }
    return launch_status();
}

// Cluster size for rows of ld keys: slices within the per-CTA cap, and enough
// CTAs to fill the GPU.
int cluster_size(int64_t ld, int64_t rows, int sms, int* slice) {
    auto slice_of = [&](int c) { return static_cast<int>(((ld + c - 1) / c + 3) / 4 * 4); };
    int C = 1;
    while (C < kMaxCluster &&
           (slice_of(C) > kSliceCap || (rows * C < 2 * sms && slice_of(2 * C) >= 2048)))
        C *= 2;
    *slice = ld > 0 ? slice_of(C) : 4;
    return C;
}

template <bool HIST>
int launch_cluster(TopkArgs a, const RowsArgs& f, int sms, cudaStream_t s) {
    const int C = cluster_size(a.ld, a.rows, sms, &a.slice);
    const int64_t max_clusters = static_cast<int64_t>(sms) * 3 / C;
    const int64_t clusters = a.rows < max_clusters ? a.rows : max_clusters;
    const int per_needed = (a.slice + kThreads - 1) / kThreads;
    if (per_needed <= 4) return launch_per<4, HIST>(a, f, C, clusters, s);
    if (per_needed <= 8) return launch_per<8, HIST>(a, f, C, clusters, s);
    if (per_needed <= 16) return launch_per<16, HIST>(a, f, C, clusters, s);
    if (per_needed <= 32) return launch_per<32, HIST>(a, f, C, clusters, s);
    return launch_per<64, HIST>(a, f, C, clusters, s);
}

void set_block_size(TopkArgs& a, int block_size) {
    a.block_size = block_size;
    a.bs_shift = (block_size & (block_size - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(block_size)) : -1;
}

}  // namespace

// The selection that follows a histogram logits kernel (see common.cuh).
int select_after_logits(const SelectRows& q, cudaStream_t s) {
    const int sms = num_sms();
    if (sms <= 0) return IX_ERR_CUDA;
    TopkArgs a{};
    RowsArgs f{};
    a.logits = q.logits;
    a.ld = q.ld;
    a.rows = q.rows;
    f.geom = q.row_len ? kRowsGiven : (q.context_lens ? kRowsDecode : kRowsPrefill);
    a.row_len = q.row_len;
    f.context_lens = q.context_lens;
    f.next_n = q.next_n;
    f.ks = q.ks;
    f.ke = q.ke;
    f.tk = q.tk;
    a.row_req = q.row_req;
    a.bt = q.block_table;
    a.bt_stride = q.bt_stride;
    set_block_size(a, q.block_size);
    a.k = q.k;
    a.out_local = q.out_local;
    a.out_global = q.out_global;
    f.hist = q.hist;
    f.status = q.status;
    if (a.rows == 0) return IX_OK;
    if (a.ld <= kSelMaxLd && a.rows >= 2 * static_cast<int64_t>(sms)) {
        const int64_t cap = static_cast<int64_t>(sms) * 6;  // 6 CTAs of 8 warps per SM
        const unsigned grid = static_cast<unsigned>((a.rows + kSelWarps - 1) / kSelWarps < cap
                                                        ? (a.rows + kSelWarps - 1) / kSelWarps
                                                        : cap);
        select_warp_kernel<<<grid, kSelWarps * 32, 0, s>>>(a, f);
        return launch_status();
    }
    return launch_cluster<true>(a, f, sms, s);
}

}  // namespace dsix

using namespace dsix;

extern "C" int ix_topk_to_global(const float* logits, int64_t ld, int64_t rows,
                                 const int32_t* row_len, const int32_t* row_req,
                                 const int32_t* block_table, int64_t bt_stride, int block_size,
                                 int k, int32_t* out_local, int32_t* out_global,
                                 ix_stream_t stream) {
    if (ld < 0 || rows < 0 || bt_stride < 0) return IX_ERR_SHAPE;
    if (k < 1 || block_size < 1) return IX_ERR_UNSUPPORTED;
    if (rows == 0) return IX_OK;
    if (ld % 4 != 0 || ld > kTopkMaxLd) return IX_ERR_UNSUPPORTED;
    if (!row_len || !row_req || !block_table || !out_global || (ld > 0 && !logits))
        return IX_ERR_NULL;
    if (ld > 0 && !aligned16(logits)) return IX_ERR_ALIGN;
    const int sms = num_sms();
    if (sms <= 0) return IX_ERR_CUDA;
    TopkArgs a{};
    a.logits = logits;
    a.ld = ld;
    a.rows = rows;
    a.row_len = row_len;
    a.row_req = row_req;
    a.bt = block_table;
    a.bt_stride = bt_stride;
    set_block_size(a, block_size);
    a.k = k;
    a.out_local = out_local;
    a.out_global = out_global;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ld <= kBlkMaxLd && rows >= 2 * static_cast<int64_t>(sms)) {
        // resident CTAs per SM: 4 at PER = 32 (registers bounded to 64), 2 at PER = 64
        const int64_t cap = static_cast<int64_t>(sms) * (ld <= kBlkThreads * 32 ? 4 : 2);
        const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
        if (ld <= kBlkThreads * 32)
            topk_block_kernel<32><<<grid, kBlkThreads, 0, s>>>(a);
        else
            topk_block_kernel<64><<<grid, kBlkThreads, 0, s>>>(a);
        return launch_status();
    }
    RowsArgs f{};
    f.geom = kRowsGiven;
    return launch_cluster<false>(a, f, sms, s);
}

extern "C" int ix_topk_from_hist(const float* logits, int64_t ld, int64_t rows, const int32_t* row_len,
                                 const int32_t* row_req, const int32_t* block_table, int64_t bt_stride,
                                 int block_size, int k, int32_t* out_local, int32_t* out_global,
                                 void* workspace, size_t workspace_bytes, ix_stream_t stream) {
    if (ld < 0 || rows < 0 || bt_stride < 0) return IX_ERR_SHAPE;
    if (k < 1 || block_size < 1) return IX_ERR_UNSUPPORTED;
    if (rows == 0) return IX_OK;
    if (ld % 4 != 0 || ld > kTopkMaxLd) return IX_ERR_UNSUPPORTED;
    if (!row_len || !row_req || !block_table || !out_global || (ld > 0 && !logits)) return IX_ERR_NULL;
    if (ld > 0 && !aligned16(logits)) return IX_ERR_ALIGN;
    if (!workspace || workspace_bytes < static_cast<size_t>(rows) * kHistRowWords * 4) return IX_ERR_WORKSPACE;
    if (!aligned16(workspace)) return IX_ERR_ALIGN;
    int* st = status_ptr();
    if (!st) return IX_ERR_CUDA;
    SelectRows q{};
    q.logits = logits;
    q.ld = ld;
    q.rows = rows;
    q.row_len = row_len;
    q.row_req = row_req;
    q.block_table = block_table;
    q.bt_stride = bt_stride;
    q.block_size = block_size;
    q.k = k;
    q.out_local = out_local;
    q.out_global = out_global;
    q.hist = static_cast<uint32_t*>(workspace);
    q.status = st;
    return select_after_logits(q, reinterpret_cast<cudaStream_t>(stream));
}
