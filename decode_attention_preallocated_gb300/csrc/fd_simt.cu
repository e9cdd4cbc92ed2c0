// fd_simt.cu -- CUDA-core decode kernel: every mode (dense prefix, causal
// window, index gather, paged cache, int8 cache, masked prefix with
// chunk skipping), head_dim 128 and 256.
//
// One thread block walks a contiguous range of 32-position tiles chosen by
// the balanced split partitioner (fd_internal.h).  Per tile it stages K and
// V in shared memory, computes the scores of every packed query row of the
// segment (GQA heads x window rows) against the tile, runs one step of the
// online softmax, and accumulates P.V in registers.  A segment that spans
// several blocks is finished by the last block to arrive (comfy-kitchen
// #239, "GQA decode": splits combined inside the same launch).
#include <cuda_runtime.h>

#include <atomic>

#include "fd_device.cuh"
#include "fd_launch.h"

namespace fd {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int T = 32;          // cache positions per tile

template <int D>
struct Layout {
    static constexpr int KST = D + 8;                 // padded K/V row (bf16)
    static constexpr int PV_CG = D / 8;               // threads across one row
    static constexpr int PV_RG = kThreads / PV_CG;    // row groups
    static constexpr int PV_RMAX = (64 + PV_RG - 1) / PV_RG;
    static constexpr int QK_RMAX = 64 / kWarps;
    static size_t smem_bytes(int rows) {
        return (size_t)rows * D * 4          // Q (fp32)
               + 2 * (size_t)T * KST * 2     // K, V tiles (bf16)
               + 3 * (size_t)T * 8           // positions, K and V row offsets (int64,
                                             // 8-byte aligned here)
               + (size_t)rows * (T + 1) * 4  // P
               + 5 * (size_t)T * 4           // k scale, v scale, valid, appended, bias
               + 6 * (size_t)T * 4           // masked mode: mask of each query row
               + 3 * (size_t)rows * 4;       // m, l, alpha
    }
};

__device__ __forceinline__ void unpack8(const uint4 &w, float *f) {
    f[0] = bf16lo(w.x); f[1] = bf16hi(w.x);
    f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    f[4] = bf16lo(w.z); f[5] = bf16hi(w.z);
    f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

// int8 code -> bf16 bits (exact: |code| <= 128 needs 8 significant bits).
__device__ __forceinline__ uint32_t i8pair_to_bf16x2(int lo, int hi) {
    return pack_bf16x2((float)lo, (float)hi);
}

template <int D>
__device__ __forceinline__ void simt_body(const Params &p) {
    using Ly = Layout<D>;
    extern __shared__ __align__(16) unsigned char smem[];
    const int rows = p.rows;
    // Q, K and V sizes are multiples of 16 bytes, so the int64 positions
    // that follow them are aligned whatever the row count.
    float *Qs = reinterpret_cast<float *>(smem);
    uint16_t *Ks = reinterpret_cast<uint16_t *>(Qs + rows * D);
    uint16_t *Vs = Ks + T * Ly::KST;
    int64_t *tpos = reinterpret_cast<int64_t *>(Vs + T * Ly::KST);
    int64_t *tko = tpos + T, *tvo = tko + T;   // element offsets of the K / V rows
    float *Ps = reinterpret_cast<float *>(tvo + T);
    float *ksc = Ps + rows * (T + 1);
    float *vsc = ksc + T;
    int *tval = reinterpret_cast<int *>(vsc + T);
    int *tnew = tval + T;                      // fused append: the row comes from k_new / v_new
    float *tbias = reinterpret_cast<float *>(tnew + T);   // gather: entry bias (log2 units)
    float *tmask = tbias + T;   // masked: [n_q][T] mask (log2 units), -inf outside the window
    float *m_s = tmask + 6 * T;
    float *l_s = m_s + rows;
    float *a_s = l_s + rows;

    __shared__ int64_t sh_total, sh_seg, sh_first, sh_n;
    __shared__ int sh_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;

    if (warp == 0) {
        int64_t tot = total_tiles_warp(p);
        if (lane == 0) sh_total = tot;
    }
    __syncthreads();
    const int64_t total = sh_total;

    // Segments with nothing to attend still need their output rows zeroed.
    for (int64_t s = c; s < p.nseg; s += G)
        if (seg_tiles(p, s) == 0) zero_segment(p, s);
    if (total == 0) return;

    const int32_t Gw = working_blocks(total, G);
    if (c >= Gw) return;
    const Split sp{total, Gw};
    const int64_t t_begin = sp.start(c), t_end = sp.start(c + 1);

    // PV ownership: thread -> 8 dims of up to PV_RMAX rows.
    const int cg = tid % Ly::PV_CG, rg = tid / Ly::PV_CG;

    int64_t t = t_begin;
    while (t < t_end) {
        __syncthreads();
        if (warp == 0) {
            SegPos pos;
            int64_t s = seg_of_tile_warp(p, t, &pos);
            if (lane == 0) { sh_seg = s; sh_first = pos.first; sh_n = pos.ntiles; }
        }
        __syncthreads();
        const int64_t s = sh_seg, first = sh_first, nt = sh_n;
        if (s < 0 || nt <= 0) break;   // cannot happen for t < total
        const int64_t piece_end = min(t_end, first + nt);
        const int c_first = sp.owner(first), c_last = sp.owner(first + nt - 1);
        const int npieces = c_last - c_first + 1;

        // Segment geometry.
        const RowMap m0 = row_of(p, s, 0);
        const int b = m0.b;
        const int hk = (int)(s % p.Hkv);
        const int64_t len = p.mode == kGather ? (int64_t)p.idx_len : seq_len(p, b);
        const int32_t *list = p.mode == kGather
                                  ? p.idx + ((int64_t)b * p.n_q + m0.i) * p.idx_len
                                  : nullptr;

        // Q rows of the segment (fp32) and fresh softmax state.
        for (int e = tid; e < rows * D; e += kThreads) {
            const int r = e / D, dd = e % D;
            const RowMap m = row_of(p, s, r);
            const uint16_t bits = p.q[(int64_t)m.b * p.qs[0] + (int64_t)m.i * p.qs[1] +
                                      (int64_t)m.h * p.qs[2] + dd];
            Qs[e] = __uint_as_float((uint32_t)bits << 16);
        }
        if (tid < rows) { m_s[tid] = neg_inf(); l_s[tid] = 0.f; a_s[tid] = 1.f; }

        float O[Ly::PV_RMAX][8];
#pragma unroll
        for (int k = 0; k < Ly::PV_RMAX; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) O[k][e] = 0.f;

        const char *kbase = reinterpret_cast<const char *>(p.k);
        const char *vbase = reinterpret_cast<const char *>(p.v);

        for (int64_t tt = t - first; tt < piece_end - first; ++tt) {
            const int64_t j0 = tt * T;
            const int ntok = (int)min((int64_t)T, len - j0);
            __syncthreads();   // previous tile fully consumed
            int live = 0;
            if (tid < T) {
                int64_t pos = j0 + tid;
                int ok = tid < ntok;
                float bias = 0.f;
                if (ok && list) {
                    const int64_t cell = list[pos];
                    if (cell >= p.cap) atomicOr(p.status, kDevBadIndex);
                    if (p.bias) bias = p.bias[((int64_t)b * p.n_q + m0.i) * p.idx_len + pos];
                    ok = cell >= 0 && cell < p.cap && bias != neg_inf();
                    pos = cell;
                }
                tbias[tid] = bias * 1.4426950408889634f;
                // Where the position's row lives: (sequence, kv head, position)
                // of a flat cache, (page, kv head, row in page) of a paged one.
                int64_t o0 = b, o2 = pos;
                if (ok && p.mode == kPaged) {
                    const int32_t pg = page_of(p, b, (int32_t)pos);
                    ok = pg >= 0;
                    o0 = pg;
                    o2 = page_row(p, (int32_t)pos);
                }
                tpos[tid] = ok ? pos : 0;
                tval[tid] = ok;
                tko[tid] = o0 * p.ks[0] + (int64_t)hk * p.ks[1] + o2 * p.ks[2];
                tvo[tid] = o0 * p.vs[0] + (int64_t)hk * p.vs[1] + o2 * p.vs[2];
                // Fused append: positions from the old length on are row
                // pos - base of k_new / v_new (this block, which owns the
                // tile, also writes them into the caches).
                int isnew = 0;
                if (ok && p.n_new > 0) {
                    const int64_t base = append_base(p, b);
                    if (pos >= base) {
                        isnew = 1;
                        tko[tid] = (int64_t)b * p.kns[0] + (pos - base) * p.kns[1] + (int64_t)hk * p.kns[2];
                        tvo[tid] = (int64_t)b * p.vns[0] + (pos - base) * p.vns[1] + (int64_t)hk * p.vns[2];
                    }
                }
                tnew[tid] = isnew;
                float kscale = 1.f, vscale = 1.f;
                if (ok && p.kv_int8) {
                    kscale = p.k_scale[o0 * p.kss[0] + (int64_t)hk * p.kss[1] + o2 * p.kss[2]];
                    vscale = p.v_scale[o0 * p.vss[0] + (int64_t)hk * p.vss[1] + o2 * p.vss[2]];
                }
                ksc[tid] = kscale;
                vsc[tid] = vscale;
                // Masked mode: each query row's mask value at this position
                // (-inf where it hides the position or the window does).
                if (p.mode == kMasked) {
                    for (int i = 0; i < p.n_q; ++i) {
                        float mv = neg_inf();
                        if (ok && (!p.causal || pos <= len - p.n_q + i))
                            mv = p.mask[(int64_t)b * p.ms[0] + (int64_t)i * p.ms[1] + pos];
                        tmask[i * T + tid] = mv == neg_inf() ? neg_inf() : mv * 1.4426950408889634f;
                        live |= mv != neg_inf();
                    }
                }
            }
            // A tile the mask hides entirely is skipped: no K / V read.
            if (__syncthreads_or(live) == 0 && p.mode == kMasked) continue;
            // Stage the K and V rows (zeros for positions that are not visible).
            if (!p.kv_int8) {
                constexpr int CPR = D / 8;   // 16-byte chunks per row
                for (int e = tid; e < 2 * T * CPR; e += kThreads) {
                    const int which = e / (T * CPR);
                    const int jj = (e / CPR) % T, cc = e % CPR;
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (tval[jj] && tnew[jj]) {
                        const uint16_t *src = (which ? p.v_new + tvo[jj] : p.k_new + tko[jj]) + cc * 8;
                        w = *reinterpret_cast<const uint4 *>(src);
                        const int64_t *cs = which ? p.vs : p.ks;
                        uint16_t *cache = const_cast<uint16_t *>(
                            static_cast<const uint16_t *>(which ? p.v : p.k));
                        *reinterpret_cast<uint4 *>(cache + (int64_t)b * cs[0] + (int64_t)hk * cs[1] +
                                                   tpos[jj] * cs[2] + cc * 8) = w;
                    } else if (tval[jj]) {
                        const char *src = which ? vbase + (tvo[jj] + cc * 8) * 2
                                                : kbase + (tko[jj] + cc * 8) * 2;
                        w = ldg_stream(src);
                    }
                    uint16_t *dst = (which ? Vs : Ks) + jj * Ly::KST + cc * 8;
                    *reinterpret_cast<uint4 *>(dst) = w;
                }
            } else {
                constexpr int CPR = D / 16;
                for (int e = tid; e < 2 * T * CPR; e += kThreads) {
                    const int which = e / (T * CPR);
                    const int jj = (e / CPR) % T, cc = e % CPR;
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (tval[jj]) {
                        const char *src = which ? vbase + (tvo[jj] + cc * 16)
                                                : kbase + (tko[jj] + cc * 16);
                        w = ldg_stream(src);
                    }
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
                    uint32_t o[8];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int8_t *by = reinterpret_cast<const int8_t *>(&ws[q4]);
                        o[2 * q4] = i8pair_to_bf16x2(by[0], by[1]);
                        o[2 * q4 + 1] = i8pair_to_bf16x2(by[2], by[3]);
                    }
                    uint16_t *dst = (which ? Vs : Ks) + jj * Ly::KST + cc * 16;
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<uint4 *>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
            __syncthreads();

            // Scores: warp w owns rows w, w+8, ...; lane = position in tile.
            float acc[Ly::QK_RMAX];
#pragma unroll
            for (int k = 0; k < Ly::QK_RMAX; ++k) acc[k] = 0.f;
#pragma unroll 4
            for (int cc = 0; cc < D / 8; ++cc) {
                float kf[8];
                unpack8(*reinterpret_cast<const uint4 *>(Ks + lane * Ly::KST + cc * 8), kf);
#pragma unroll
                for (int k = 0; k < Ly::QK_RMAX; ++k) {
                    const int r = warp + kWarps * k;
                    if (r < rows) {
                        const float4 qa = *reinterpret_cast<const float4 *>(Qs + r * D + cc * 8);
                        const float4 qb = *reinterpret_cast<const float4 *>(Qs + r * D + cc * 8 + 4);
                        acc[k] += qa.x * kf[0] + qa.y * kf[1] + qa.z * kf[2] + qa.w * kf[3] +
                                  qb.x * kf[4] + qb.y * kf[5] + qb.z * kf[6] + qb.w * kf[7];
                    }
                }
            }
            // Mask and one online-softmax step per row (same warp owns the row).
#pragma unroll
            for (int k = 0; k < Ly::QK_RMAX; ++k) {
                const int r = warp + kWarps * k;
                if (r < rows) {
                    bool vis = tval[lane] != 0;
                    if (p.causal && p.mode != kGather) {
                        const int i = r % p.n_q;
                        vis = vis && tpos[lane] <= len - p.n_q + i;
                    }
                    float mb = 0.f;
                    if (p.mode == kMasked) {
                        mb = tmask[(r % p.n_q) * T + lane];
                        vis = vis && mb != neg_inf();
                    }
                    const float sc = vis ? acc[k] * ksc[lane] * p.scale_log2 + tbias[lane] + mb
                                         : neg_inf();
                    float tmax = sc;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
                    const float m_old = m_s[r];
                    const float m_new = fmaxf(m_old, tmax);
                    const float m_use = m_new == neg_inf() ? 0.f : m_new;
                    const float alpha = fast_exp2(m_old - m_use);
                    const float pr = vis ? fast_exp2(sc - m_use) : 0.f;
                    float psum = pr;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        psum += __shfl_xor_sync(0xffffffffu, psum, o);
                    Ps[r * (T + 1) + lane] = pr * vsc[lane];
                    __syncwarp();
                    if (lane == 0) {
                        m_s[r] = m_new;
                        l_s[r] = l_s[r] * alpha + psum;
                        a_s[r] = alpha;
                    }
                }
            }
            __syncthreads();

            // O = alpha * O + P . V
#pragma unroll
            for (int k = 0; k < Ly::PV_RMAX; ++k) {
                const int r = rg + Ly::PV_RG * k;
                if (r < rows) {
                    const float a = a_s[r];
#pragma unroll
                    for (int e = 0; e < 8; ++e) O[k][e] *= a;
                }
            }
            for (int jj = 0; jj < ntok; ++jj) {
                float vf[8];
                unpack8(*reinterpret_cast<const uint4 *>(Vs + jj * Ly::KST + cg * 8), vf);
#pragma unroll
                for (int k = 0; k < Ly::PV_RMAX; ++k) {
                    const int r = rg + Ly::PV_RG * k;
                    if (r < rows) {
                        const float pw = Ps[r * (T + 1) + jj];
#pragma unroll
                        for (int e = 0; e < 8; ++e) O[k][e] += pw * vf[e];
                    }
                }
            }
        }
        __syncthreads();

        // ---- finish the piece
        if (npieces == 1) {
#pragma unroll
            for (int k = 0; k < Ly::PV_RMAX; ++k) {
                const int r = rg + Ly::PV_RG * k;
                if (r < rows) {
                    const float l = l_s[r];
                    const float inv = l > 0.f ? 1.f / l : 0.f;
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = O[k][e] * inv;
                    store_out8(p, row_of(p, s, r), cg * 8, o);
                }
            }
        } else {
            float *slot = slot_ptr(p, s, c);
#pragma unroll
            for (int k = 0; k < Ly::PV_RMAX; ++k) {
                const int r = rg + Ly::PV_RG * k;
                if (r < rows) {
                    float4 *dst = reinterpret_cast<float4 *>(slot + r * D + cg * 8);
                    dst[0] = make_float4(O[k][0], O[k][1], O[k][2], O[k][3]);
                    dst[1] = make_float4(O[k][4], O[k][5], O[k][6], O[k][7]);
                }
            }
            if (tid < rows) {
                slot[rows * D + tid] = m_s[tid];
                slot[rows * D + rows + tid] = l_s[tid];
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int old = atomicAdd(p.counters + s, 1);
                sh_last = old == npieces - 1;
            }
            __syncthreads();
            if (sh_last) {
                __threadfence();
                // Merge the pieces' partials in one pass per row: running
                // maximum, merged sum and accumulator rescaled as each piece
                // arrives.  Rows are clamped into range (weight 0 beyond
                // `rows`), so every load is unconditional and one piece's loads
                // are all in flight together.
                int rr[Ly::PV_RMAX];
                float M[Ly::PV_RMAX], Ls[Ly::PV_RMAX], o[Ly::PV_RMAX][8];
#pragma unroll
                for (int k = 0; k < Ly::PV_RMAX; ++k) {
                    const int r = rg + Ly::PV_RG * k;
                    rr[k] = r < rows ? r : rows - 1;
                    M[k] = neg_inf();
                    Ls[k] = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[k][e] = 0.f;
                }
#pragma unroll 2
                for (int c2 = c_first; c2 <= c_last; ++c2) {
                    const float *sl = slot_ptr(p, s, c2);
#pragma unroll
                    for (int k = 0; k < Ly::PV_RMAX; ++k) {
                        const float mv = __ldcg(sl + rows * D + rr[k]);
                        const float lv = __ldcg(sl + rows * D + rows + rr[k]);
                        const float4 a4 = __ldcg(reinterpret_cast<const float4 *>(sl + rr[k] * D + cg * 8));
                        const float4 b4 = __ldcg(reinterpret_cast<const float4 *>(sl + rr[k] * D + cg * 8 + 4));
                        const float mn = fmaxf(M[k], mv);
                        const float mu = mn == neg_inf() ? 0.f : mn;
                        const float a = fast_exp2(M[k] - mu), w = fast_exp2(mv - mu);
                        M[k] = mn;
                        Ls[k] = Ls[k] * a + w * lv;
                        const float v[8] = {a4.x, a4.y, a4.z, a4.w, b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[k][e] = o[k][e] * a + w * v[e];
                    }
                }
#pragma unroll
                for (int k = 0; k < Ly::PV_RMAX; ++k) {
                    const int r = rg + Ly::PV_RG * k;
                    if (r < rows) {
                        const float inv = Ls[k] > 0.f ? 1.f / Ls[k] : 0.f;
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[k][e] *= inv;
                        store_out8(p, row_of(p, s, r), cg * 8, o[k]);
                    }
                }
                if (tid == 0) p.counters[s] = 0;
            }
        }
        t = piece_end;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads)
simt_kernel(const __grid_constant__ Params p) {
    simt_body<D>(p);
    if (p.n_new > 0) append_exit(p);
}

template <int D>
int launch_d(const Params &p, int G, cudaStream_t st) {
    const size_t smem = Layout<D>::smem_bytes(p.rows);
    // the dynamic shared memory opt-in (for the largest row count), once per
    // device
    static std::atomic<uint64_t> opted{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -5;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
        const size_t most = Layout<D>::smem_bytes(64) > smem ? Layout<D>::smem_bytes(64) : smem;
        if (cudaFuncSetAttribute(simt_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)most) != cudaSuccess)
            return -5;
        opted.fetch_or(bit, std::memory_order_release);
    }
    simt_kernel<D><<<G, kThreads, smem, st>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace

int simt_tile_tokens() { return T; }

int launch_simt(const Params &p, int G, cudaStream_t st) {
    if (p.d == 128) return launch_d<128>(p, G, st);
    if (p.d == 256) return launch_d<256>(p, G, st);
    return -2;
}

}  // namespace fd
