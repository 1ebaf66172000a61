// topk.cu -- per-row top-k of the indexer logits + remap to global paged-KV slots.
//
// Selection: radix select on an order-preserving 32-bit key of each logit
// (-0.0 folded onto +0.0), three digit passes of 11/11/10 bits over the
// row, then one ordered compaction pass that keeps every key above the
// threshold and the lowest-indexed keys equal to it.  Output is in ascending
// index order, so equal values resolve to the lower index and the result is
// unique.
//
// Layout on the GPU: a row is split across a thread-block cluster of C CTAs
// (C = 1, 2, 4 or 8, picked on the host from the row length and row count).
// Each CTA keeps its contiguous slice of the row in shared memory (read from
// HBM once, 16-byte loads).  Per pass, CTAs build a local histogram and add
// it into rank 0's histogram through distributed shared memory; after a
// cluster barrier every CTA reads the merged histogram and picks the same
// digit.  The ordered compaction needs each CTA's count of kept keys before
// its slice, exchanged the same way.  No global scratch, no atomics on HBM, no
// waiting on other clusters.
#include <cooperative_groups.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsix {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxCluster = 8;
constexpr int kSliceCap = 32768;  // keys per CTA slice (128 KB of shared memory)
constexpr int kBins0 = 2048, kBins1 = 2048, kBins2 = 1024;
constexpr int kMergedInts = kBins0 + kBins1 + kBins2;

struct TopkArgs {
    const float* logits;
    int64_t ld;
    int64_t rows;
    const int32_t* row_len;
    const int32_t* row_req;
    const int32_t* bt;
    int64_t bt_stride;
    int block_size;
    int k;
    int32_t* out_local;
    int32_t* out_global;
    int slice;  // keys per CTA (multiple of 4)
};

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;  // -0.0 == +0.0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ void emit(const TopkArgs& a, int64_t r, int b, int pos, int s) {
    int32_t g = -1;
    if (s >= 0) {
        const int64_t blk = __ldg(a.bt + static_cast<int64_t>(b) * a.bt_stride + s / a.block_size);
        g = static_cast<int32_t>(blk * a.block_size + s % a.block_size);
    }
    if (a.out_local) a.out_local[r * a.k + pos] = s;
    a.out_global[r * a.k + pos] = g;
}

// Block-wide exclusive scan (kThreads threads).  *total = sum.
__device__ __forceinline__ int scan_excl(int v, int* scratch, int* total) {
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
        const int s = lane < nw ? scratch[lane] : 0;
        int inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < nw) scratch[32 + lane] = inc - s;
        if (lane == nw - 1) scratch[64] = inc;
    }
    __syncthreads();
    const int r = scratch[32 + warp] + x - v;
    *total = scratch[64];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x;

    extern __shared__ __align__(16) uint8_t smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);                       // [slice]
    int* local = reinterpret_cast<int*>(smem + static_cast<size_t>(a.slice) * 4);  // [2048]
    int* merged = local + kBins0;                                               // [2][kMergedInts]
    int* counts = merged + 2 * kMergedInts;                                     // [2][kMaxCluster][2]
    int* scratch = counts + 2 * kMaxCluster * 2;                                // [72]
    int* pick = scratch + 72;                                                   // [3]

    for (int i = tid; i < kBins0; i += kThreads) local[i] = 0;
    if (rank == 0)
        for (int i = tid; i < 2 * kMergedInts; i += kThreads) merged[i] = 0;
    cluster.sync();

    int* merged0 = cluster.map_shared_rank(merged, 0);
    int* counts0 = cluster.map_shared_rank(counts, 0);

    const int64_t cid = blockIdx.x / C;
    const int64_t nclusters = gridDim.x / C;
    int nt = 0;  // non-trivial rows processed (selects the double buffer)
    for (int64_t r = cid; r < a.rows; r += nclusters) {
        int64_t L = __ldg(a.row_len + r);
        L = L < 0 ? 0 : (L > a.ld ? a.ld : L);
        const int b = __ldg(a.row_req + r);
        if (L <= a.k) {
            for (int i = rank * kThreads + tid; i < a.k; i += C * kThreads)
                emit(a, r, b, i, i < L ? i : -1);
            continue;
        }
        const int P = nt & 1;
        ++nt;
        int* mP0 = merged0 + P * kMergedInts;  // rank 0's, through DSMEM
        int* cP0 = counts0 + P * kMaxCluster * 2;
        const int lo = rank * a.slice;
        const int64_t avail = L - lo;
        const int n = avail <= 0 ? 0 : static_cast<int>(avail < a.slice ? avail : a.slice);
        const float* src = a.logits + r * a.ld + lo;

        uint32_t prefix = 0;
        int k_rem = a.k;
        int shift = 32;  // keys compare on u >> shift against prefix (32: all equal)
        int moff = 0;
        bool done = false;
        for (int p = 0; p < 3 && !done; ++p) {
            const int nbits = p < 2 ? 11 : 10;
            const int nb = 1 << nbits;
            const int sh = shift - nbits;
            // ---- local histogram of the next digit among keys matching the prefix
            if (p == 0) {
                for (int i = tid * 4; i < n; i += kThreads * 4) {
                    if (i + 4 <= n) {
                        const float4 v = __ldg(reinterpret_cast<const float4*>(src + i));
                        const uint32_t u0 = order_key(v.x), u1 = order_key(v.y);
                        const uint32_t u2 = order_key(v.z), u3 = order_key(v.w);
                        *reinterpret_cast<uint4*>(keys + i) = make_uint4(u0, u1, u2, u3);
                        atomicAdd(local + (u0 >> sh), 1);
                        atomicAdd(local + (u1 >> sh), 1);
                        atomicAdd(local + (u2 >> sh), 1);
                        atomicAdd(local + (u3 >> sh), 1);
                    } else {
                        for (int j = i; j < n; ++j) {
                            const uint32_t u = order_key(__ldg(src + j));
                            keys[j] = u;
                            atomicAdd(local + (u >> sh), 1);
                        }
                    }
                }
            } else {
                for (int i = tid; i < n; i += kThreads) {
                    const uint32_t u = keys[i];
                    if ((u >> shift) == prefix) atomicAdd(local + ((u >> sh) & (nb - 1)), 1);
                }
            }
            __syncthreads();
            for (int i = tid; i < nb; i += kThreads) {
                const int c = local[i];
                if (c) {
                    atomicAdd(mP0 + moff + i, c);
                    local[i] = 0;
                }
            }
            if (p == 0 && rank == 0) {
                // the other buffer was last read before this row began
                int* other = merged + (P ^ 1) * kMergedInts;
                for (int i = tid; i < kMergedInts; i += kThreads) other[i] = 0;
            }
            cluster.sync();
            // ---- pick the digit holding the k_rem-th largest key (bins high to low)
            const int per = nb / kThreads;
            const int top = nb - 1 - tid * per;
            int c[4];
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c[i] = i < per ? mP0[moff + top - i] : 0;
                sum += c[i];
            }
            int total;
            const int above = scan_excl(sum, scratch, &total);
            if (above < k_rem && above + sum >= k_rem) {
                int acc = above;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < per && acc + c[i] >= k_rem) {
                        pick[0] = top - i;
                        pick[1] = acc;
                        pick[2] = c[i];
                        break;
                    }
                    acc += c[i];
                }
            }
            __syncthreads();
            const int digit = pick[0];
            k_rem -= pick[1];
            prefix = (shift == 32 ? 0u : (prefix << nbits)) | static_cast<uint32_t>(digit);
            shift = sh;
            moff += nb;
            done = (pick[2] == k_rem);  // every key in this bin is kept
            __syncthreads();
        }
        // keys with (u >> shift) > prefix are kept; of those == prefix, the first k_rem.
        // ---- per-CTA counts, exchanged through rank 0
        int gt = 0, eq = 0;
        for (int i = tid; i < n; i += kThreads) {
            const uint32_t v = keys[i] >> shift;
            gt += v > prefix;
            eq += v == prefix;
        }
        // n <= 32768, so each count fits a 16-bit field (unpacked as unsigned)
        const int packed = static_cast<int>((static_cast<uint32_t>(gt) << 16) | static_cast<uint32_t>(eq));
        int tot;
        scan_excl(packed, scratch, &tot);
        if (tid == 0) {
            cP0[2 * rank] = static_cast<int>(static_cast<uint32_t>(tot) >> 16);
            cP0[2 * rank + 1] = static_cast<int>(static_cast<uint32_t>(tot) & 0xFFFFu);
        }
        cluster.sync();
        int carry_gt = 0, carry_eq = 0;
        for (int j = 0; j < rank; ++j) {
            carry_gt += cP0[2 * j];
            carry_eq += cP0[2 * j + 1];
        }
        // ---- ordered compaction: 4 consecutive keys per thread per chunk
        for (int base = 0; base < n; base += kThreads * 4) {
            const int i0 = base + tid * 4;
            int fg[4], fe[4];
            int tg = 0, te = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool in = i0 + j < n;
                const uint32_t v = in ? keys[i0 + j] >> shift : 0u;
                fg[j] = in && v > prefix;
                fe[j] = in && v == prefix;
                tg += fg[j];
                te += fe[j];
            }
            int chunk;
            const int ex = scan_excl((tg << 16) | te, scratch, &chunk);
            int bg = carry_gt + static_cast<int>(static_cast<uint32_t>(ex) >> 16);
            int be = carry_eq + (ex & 0xFFFF);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool keep = fg[j] || (fe[j] && be < k_rem);
                const int pos = bg + min(be, k_rem);
                if (keep && pos < a.k) emit(a, r, b, pos, lo + i0 + j);
                bg += fg[j];
                be += fe[j];
            }
            carry_gt += static_cast<int>(static_cast<uint32_t>(chunk) >> 16);
            carry_eq += chunk & 0xFFFF;
        }
    }
    cluster.sync();  // no CTA leaves while others may still read its shared memory
}

size_t smem_bytes(int slice) {
    return static_cast<size_t>(slice) * 4 + (kBins0 + 2 * kMergedInts + 2 * kMaxCluster * 2 + 72 + 4) * 4;
}

}  // namespace
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
    if (ld % 4 != 0 || ld > static_cast<int64_t>(kMaxCluster) * kSliceCap) return IX_ERR_UNSUPPORTED;
    if (!row_len || !row_req || !block_table || !out_global || (ld > 0 && !logits))
        return IX_ERR_NULL;
    if (ld > 0 && !aligned16(logits)) return IX_ERR_ALIGN;
    const int sms = num_sms();
    if (sms <= 0) return IX_ERR_CUDA;
    // cluster size: enough CTAs to cover the GPU, slices no longer than the cap
    int C = 1;
    auto slice_of = [&](int c) { return static_cast<int>(((ld + c - 1) / c + 3) / 4 * 4); };
    while (C < kMaxCluster &&
           (slice_of(C) > kSliceCap || (rows * C < 2 * sms && slice_of(2 * C) >= 1024)))
        C *= 2;
    const int slice = ld > 0 ? slice_of(C) : 4;
    const size_t smem = smem_bytes(slice);
    {
        static std::mutex mu;
        static std::vector<size_t> set;
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return IX_ERR_CUDA;
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= static_cast<int>(set.size())) set.resize(dev + 1, 0);
        if (set[dev] < smem) {
            if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_bytes(kSliceCap))) != cudaSuccess)
                return IX_ERR_CUDA;
            set[dev] = smem_bytes(kSliceCap);
        }
    }
    TopkArgs a{};
    a.logits = logits;
    a.ld = ld;
    a.rows = rows;
    a.row_len = row_len;
    a.row_req = row_req;
    a.bt = block_table;
    a.bt_stride = bt_stride;
    a.block_size = block_size;
    a.k = k;
    a.out_local = out_local;
    a.out_global = out_global;
    a.slice = slice;
    const int64_t max_clusters = static_cast<int64_t>(sms) * 4 / C;
    const int64_t clusters = rows < max_clusters ? rows : max_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * C));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, topk_kernel, a) != cudaSuccess) {
        cudaGetLastError();
        return IX_ERR_CUDA;
    }
    return launch_status();
}
