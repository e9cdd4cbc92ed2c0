// fd_topk.cu -- index lists for the gather mode from block scores: top-k over
// the blocks of each (sequence, query row), then only the winners expanded
// to their cells ("qwen4exp : gather-based sparse attention for QSA
// decode", llama.cpp #28213, review discussion: the selection over the full
// cell range was the cost that grew with depth; take top-k over blocks and
// expand only the winners).
//
// One thread block per row.  The row's candidate scores (blocks whose first
// cell lies below the length) become order-preserving 32-bit keys in shared
// memory; a radix select (four 8-bit digits, most significant first, one
// 256-bin shared histogram per digit) finds the k-th largest key and how many
// of the keys equal to it are taken; an ordered compaction (block-wide
// scans: per 1024-key chunk for few keys, over per-thread runs of 32 for
// many) lists the winners in increasing block order, taking equal keys by
// lowest index; the expansion writes block*size + c, or -1 past the length.
// Scores are read once from HBM; everything else stays on chip.
#include <cuda_runtime.h>

#include <atomic>

#include "fd_launch.h"

namespace fd {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kKeysPerThread = kTopkMaxBlocks / kTopkThreads;   // the compaction's run
constexpr int kChunkedMax = 8192;   // up to here the chunked compaction is faster

// Larger float -> larger key; -0 and +0 share a key, so they tie (and the
// lower index wins), as they compare equal.
__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of x over the block's threads (in thread order), and
// the block total.  Every thread of the block calls it.
__device__ __forceinline__ int block_exclusive_scan(int x, int *total, int *wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kTopkWarps ? wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kTopkWarps) wsum[lane] = wi - w;   // exclusive warp offsets
        if (lane == 31) wsum[32] = wi;                 // block total
    }
    __syncthreads();
    const int r = wsum[warp] + incl - x;
    *total = wsum[32];
    __syncthreads();   // wsum is reused by the next call
    return r;
}

struct TopkArgs {
    const float *scores;       // [rows, n_blocks]
    const int32_t *kv_lengths; // [B]
    int32_t *idx;              // [rows, top_k * block_size]
    int32_t n_q, n_blocks, block_size, top_k;
};

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const __grid_constant__ TopkArgs a) {
    extern __shared__ uint32_t keys[];   // [n_blocks]: keys, then the winners
    __shared__ uint32_t hist[256];
    __shared__ int wsum[33];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_rem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;
    const int b = (int)(row / a.n_q);
    const int64_t span = (int64_t)a.n_blocks * a.block_size;
    int64_t L = a.kv_lengths[b];
    L = L < 0 ? 0 : (L > span ? span : L);
    const int nvalid = (int)((L + a.block_size - 1) / a.block_size);

    const float *srow = a.scores + row * a.n_blocks;
    for (int j = tid; j < nvalid; j += kTopkThreads) keys[j] = order_key(__ldg(srow + j));
    __syncthreads();

    // Radix select of the k-th largest key: digit by digit, the histogram of
    // the keys that still match the chosen prefix; rem counts the keys still
    // to take among those equal to the prefix so far.
    const bool take_all = nvalid <= a.top_k;
    uint32_t kth = 0u;
    int need_eq = 0;
    if (!take_all) {
        uint32_t prefix = 0u, mask = 0u;
        if (tid == 0) sh_rem = a.top_k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
            __syncthreads();
            for (int j = tid; j < nvalid; j += kTopkThreads) {
                const uint32_t k = keys[j];
                if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 255-8l down to 248-8l
                const int rem = sh_rem;
                int s = 0;
#pragma unroll
                for (int q = 0; q < 8; ++q) s += (int)hist[255 - 8 * lane - q];
                int cum = s;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, cum, o);
                    if (lane >= o) cum += y;
                }
                const uint32_t hit = __ballot_sync(0xffffffffu, cum >= rem);
                if (lane == __ffs(hit) - 1) {
                    int acc = cum - s;   // keys in higher bins
                    for (int q = 0; q < 8; ++q) {
                        const int d = 255 - 8 * lane - q;
                        const int h = (int)hist[d];
                        if (acc + h >= rem) {
                            sh_prefix = prefix | ((uint32_t)d << shift);
                            sh_rem = rem - acc;
                            break;
                        }
                        acc += h;
                    }
                }
            }
            __syncthreads();
            prefix = sh_prefix;
            mask |= 255u << shift;
        }
        kth = prefix;
        need_eq = sh_rem;
    }

    // Ordered compaction, in place: winners are keys above the k-th, then
    // keys equal to it by lowest index, listed in increasing order.
    int nsel = 0;
    if (nvalid <= kChunkedMax) {
        // few keys: 1024-key chunks, two block-wide scans each (equal keys,
        // then winners); a winner's slot never lies after its own index
        int neq = 0;
        for (int c0 = 0; c0 < nvalid; c0 += kTopkThreads) {
            const int j = c0 + tid;
            const uint32_t k = j < nvalid ? keys[j] : 0u;
            const bool gt = j < nvalid && (take_all || k > kth);
            const bool eq = j < nvalid && !take_all && k == kth;
            int teq, tsel;
            const int eq_rank = neq + block_exclusive_scan(eq ? 1 : 0, &teq, wsum);
            const bool sel = gt || (eq && eq_rank < need_eq);
            const int pos = nsel + block_exclusive_scan(sel ? 1 : 0, &tsel, wsum);
            if (sel) keys[pos] = (uint32_t)j;
            nsel += tsel;
            neq += teq;
            __syncthreads();
        }
    } else {
        // many keys: thread t owns the run t*KPT .. t*KPT+KPT-1 (held in
        // registers), so two scans in all give every thread its place
        uint32_t run[kKeysPerThread];
        const int r0 = tid * kKeysPerThread;
        int n_eq = 0, n_gt = 0;
#pragma unroll
        for (int q = 0; q < kKeysPerThread; ++q) {
            const int j = r0 + q;
            run[q] = j < nvalid ? keys[j] : 0u;
            if (j < nvalid) {
                if (take_all || run[q] > kth) ++n_gt;
                else if (run[q] == kth) ++n_eq;
            }
        }
        int teq, tsel;
        const int eq_before = block_exclusive_scan(n_eq, &teq, wsum);
        int eq_take = need_eq - eq_before;
        eq_take = eq_take < 0 ? 0 : (eq_take > n_eq ? n_eq : eq_take);
        int pos = block_exclusive_scan(n_gt + eq_take, &tsel, wsum);   // (ends with a barrier)
        nsel = tsel;
#pragma unroll
        for (int q = 0; q < kKeysPerThread; ++q) {
            const int j = r0 + q;
            if (j < nvalid) {
                bool sel = take_all || run[q] > kth;
                if (!sel && run[q] == kth && eq_take > 0) {
                    sel = true;
                    --eq_take;
                }
                if (sel) keys[pos++] = (uint32_t)j;
            }
        }
        __syncthreads();
    }

    // Expansion: winner t covers list entries t*size .. t*size + size - 1.
    const int64_t W = (int64_t)a.top_k * a.block_size;
    int32_t *orow = a.idx + row * W;
    for (int64_t e = tid; e < W; e += kTopkThreads) {
        const int64_t t = e / a.block_size;
        int32_t v = -1;
        if (t < nsel) {
            const int64_t cell = (int64_t)keys[t] * a.block_size + (e - t * a.block_size);
            v = cell < L ? (int32_t)cell : -1;
        }
        orow[e] = v;
    }
}

}  // namespace

int topk_max_blocks() { return kTopkMaxBlocks; }

int launch_topk(const float *scores, int B, int n_q, int n_blocks, const int32_t *kv_lengths,
                int block_size, int top_k, int32_t *idx, cudaStream_t st) {
    if (n_blocks < 1 || n_blocks > kTopkMaxBlocks) return -2;
    const size_t smem = (size_t)n_blocks * 4;
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -5;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
        if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTopkMaxBlocks * 4) != cudaSuccess)
            return -5;
        opted.fetch_or(bit, std::memory_order_release);
    }
    TopkArgs a{scores, kv_lengths, idx, n_q, n_blocks, block_size, top_k};
    topk_kernel<<<(unsigned)((int64_t)B * n_q), kTopkThreads, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace fd
