// fd_device.cuh -- device helpers shared by the decode kernels: bf16/int8
// unpacking, the segment walk of the split partitioner, output stores and
// the in-launch combine of split partials.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fd_internal.h"

namespace fd {

constexpr int kDevBadLength = 1;   // mirrors FD_DEV_BAD_LENGTH
constexpr int kDevBadIndex = 2;    // mirrors FD_DEV_BAD_INDEX

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x with the SFU instruction (relative error ~2^-22; results below the
// fp32 normal range flush to 0, which only drops weights < 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two bf16 packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------- segments
// Segment s of a dense launch is (b, hk) = (s / Hkv, s % Hkv) with
// ceil(L_b / tile) tiles; a gather launch has nseg = B*n_q*Hkv segments of
// ceil(idx_len / tile) tiles each.
__device__ __forceinline__ int64_t seq_len(const Params &p, int b) {
    const int64_t raw = (int64_t)__ldg(p.kv_lengths + b);
    if (raw < 0 || raw + p.n_new > p.cap) atomicOr(p.status, kDevBadLength);
    return clamp_len(clamp_len(raw, p.cap) + p.n_new, p.cap);
}

// Fused append: position of sequence b's first appended row (its length
// before the call, clamped to [0, cap]).
__device__ __forceinline__ int64_t append_base(const Params &p, int b) {
    return clamp_len((int64_t)__ldg(p.kv_lengths + b), p.cap);
}

// Fused append, end of the launch: once every block of the grid has passed
// here (so no block reads kv_lengths any more), the last one writes the new
// lengths (if asked) and resets the launch counters for the next launch.
// Called by every thread of every block.
static __device__ __noinline__ void append_exit(const Params &p) {
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(p.grid + 1, 1) == (int)gridDim.x - 1;
        if (last) __threadfence();
    }
    __syncthreads();
    if (!last) return;
    if (p.len_update)
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
            const int64_t raw = (int64_t)p.kv_lengths[b];
            p.len_update[b] = (int32_t)clamp_len(clamp_len(raw, p.cap) + p.n_new, p.cap);
        }
    __syncthreads();
    if (threadIdx.x == 0) {
        p.grid[0] = 0;
        p.grid[1] = 0;
        __threadfence();
    }
}

// Paged caches: which page of its sequence logical position pos falls on,
// and its row in that page (shifts for power-of-two page sizes).
__device__ __forceinline__ int32_t page_slot(const Params &p, int32_t pos) {
    return p.page_shift >= 0 ? pos >> p.page_shift : pos / p.page_size;
}
__device__ __forceinline__ int32_t page_row(const Params &p, int32_t pos) {
    return p.page_shift >= 0 ? pos & (p.page_size - 1) : pos % p.page_size;
}

// The pool page that holds logical position pos (< cap) of sequence b, or
// -1, with FD_DEV_BAD_INDEX set, when the table entry names no page of the
// pool (the position is then skipped).
__device__ __forceinline__ int32_t page_of(const Params &p, int b, int32_t pos) {
    const int32_t e = __ldg(p.block_table + (int64_t)b * p.max_pages + page_slot(p, pos));
    if (e < 0 || e >= p.num_pages) {
        atomicOr(p.status, kDevBadIndex);
        return -1;
    }
    return e;
}

__device__ __forceinline__ int64_t seg_tiles(const Params &p, int64_t s) {
    if (p.mode == kGather) return ceil_div(p.idx_len, p.tile);
    return ceil_div(seq_len(p, (int)(s / p.Hkv)), p.tile);
}

// Total tile count of the launch, computed by one warp (every lane returns
// the same value).
__device__ __forceinline__ int64_t total_tiles_warp(const Params &p) {
    const int lane = threadIdx.x & 31;
    if (p.mode == kGather) return p.nseg * ceil_div(p.idx_len, p.tile);
    int64_t acc = 0;
    for (int b = lane; b < p.B; b += 32)
        acc += (int64_t)p.Hkv * ceil_div(seq_len(p, b), p.tile);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// First tile index of segment s and its tile count.  For the dense mode the
// prefix over sequences is summed by one warp.
struct SegPos {
    int64_t first;   // global index of the segment's first tile
    int64_t ntiles;
};

__device__ __forceinline__ SegPos seg_pos_warp(const Params &p, int64_t s) {
    const int lane = threadIdx.x & 31;
    if (p.mode == kGather) {
        int64_t n = ceil_div(p.idx_len, p.tile);
        return {s * n, n};
    }
    const int b = (int)(s / p.Hkv), hk = (int)(s % p.Hkv);
    int64_t acc = 0;
    for (int bb = lane; bb < b; bb += 32)
        acc += (int64_t)p.Hkv * ceil_div(seq_len(p, bb), p.tile);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    int64_t n = ceil_div(seq_len(p, b), p.tile);
    return {acc + (int64_t)hk * n, n};
}

// Segment that holds global tile t (dense: warp-parallel scan over
// sequences).  Every lane returns the same segment and its first tile.
__device__ __forceinline__ int64_t seg_of_tile_warp(const Params &p, int64_t t,
                                                    SegPos *pos) {
    const int lane = threadIdx.x & 31;
    if (p.mode == kGather) {
        int64_t n = ceil_div(p.idx_len, p.tile);
        int64_t s = t / n;
        *pos = {s * n, n};
        return s;
    }
    int64_t base = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int64_t n = b < p.B ? ceil_div(seq_len(p, b), p.tile) : 0;
        int64_t w = (int64_t)p.Hkv * n;
        int64_t incl = w;   // inclusive scan over the 32 lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        const int64_t excl = incl - w;
        const bool here = b < p.B && w > 0 && t >= base + excl && t < base + incl;
        const unsigned m = __ballot_sync(0xffffffffu, here);
        if (m) {
            const int src = __ffs(m) - 1;
            const int64_t e = __shfl_sync(0xffffffffu, excl, src);
            const int64_t nb = __shfl_sync(0xffffffffu, n, src);
            const int64_t off = t - (base + e);
            const int hk = (int)(off / nb);
            *pos = {base + e + (int64_t)hk * nb, nb};
            return (int64_t)(b0 + src) * p.Hkv + hk;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    *pos = {0, 0};
    return -1;
}

// --------------------------------------------------------------- row maps
// Query row r of segment s -> (b, i, h).  Dense rows are ordered
// (local head, query row); gather segments hold one query row.
struct RowMap {
    int b, i, h;
};

__device__ __forceinline__ RowMap row_of(const Params &p, int64_t s, int r) {
    RowMap m;
    if (p.mode == kGather) {
        const int64_t bi = s / p.Hkv;
        const int hk = (int)(s % p.Hkv);
        m.b = (int)(bi / p.n_q);
        m.i = (int)(bi % p.n_q);
        m.h = hk * p.g + r;
    } else {
        const int hk = (int)(s % p.Hkv);
        m.b = (int)(s / p.Hkv);
        m.i = r % p.n_q;
        m.h = hk * p.g + r / p.n_q;
    }
    return m;
}

// Store 8 consecutive output values of one row (dense index dd0..dd0+7).
__device__ __forceinline__ void store_out8(const Params &p, const RowMap &m,
                                           int dd0, const float *o) {
    const int64_t off = (int64_t)m.b * p.os[0] + (int64_t)m.i * p.os[1] +
                        (int64_t)m.h * p.os[2] + dd0;
    if (p.out_f32) {
        float *dst = reinterpret_cast<float *>(p.out) + off;
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[e] = o[e];
    } else {
        uint16_t *dst = reinterpret_cast<uint16_t *>(p.out) + off;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(o[2 * e], o[2 * e + 1]);
        if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dst[2 * e] = (uint16_t)(w[e] & 0xffffu);
                dst[2 * e + 1] = (uint16_t)(w[e] >> 16);
            }
        }
    }
}

// Zero every output row of segment s (segments with no tiles).
__device__ __forceinline__ void zero_segment(const Params &p, int64_t s) {
    const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int per_row = p.d / 8;
    for (int e = threadIdx.x; e < p.rows * per_row; e += blockDim.x) {
        const int r = e / per_row, c = e % per_row;
        store_out8(p, row_of(p, s, r), c * 8, z);
    }
}

// Workspace slot of piece (s, c): O[rows][d], m[rows], l[rows] (16-byte aligned).
__device__ __forceinline__ float *slot_ptr(const Params &p, int64_t s, int c) {
    return p.partials + (size_t)(s + c) * (size_t)slot_floats(p.rows, p.d);
}

}  // namespace fd
