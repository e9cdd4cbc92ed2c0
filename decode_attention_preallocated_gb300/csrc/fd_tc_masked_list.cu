// fd_tc_masked_list.cu -- the masked prefix on the tensor-core kernel with a
// chunk list: a pass over the mask lists, per sequence and in order, the
// 32-position chunks some query row sees, and the decode launch walks only
// those, four to a tile, so its work follows the visible chunks rather than
// the length ("qwen4exp : gather-based sparse attention for QSA decode",
// llama.cpp #28213, Metal measurements: the FA-vec kernel skips fully masked
// 32-cell chunks; here the skipped chunks cost no tile either).
#include "fd_tc_kernel.cuh"

namespace fd {

namespace {

constexpr int kListThreads = 256;   // 8 warps
constexpr int kListChunks = 256;    // chunks one block decides (32 per warp)
constexpr int kListMaxBlocks = 1024;   // blocks per sequence (capacity <= 2^23)
static_assert(kListChunks == kListThreads, "the last block copies one entry per thread and region");

struct ListLayout {
    int64_t mls;       // list row stride (entries)
    int64_t nblk;      // blocks of the pass per sequence
    int64_t cnt_off, stage_off, stage_cnt_off, total;   // in int32
};

ListLayout list_layout(int64_t B, int64_t cap) {
    ListLayout l;
    const int64_t nch = (cap + 31) / 32;
    l.mls = (nch + 3) / 4 * 4;
    l.nblk = (nch + kListChunks - 1) / kListChunks;
    l.cnt_off = B * l.mls;
    l.stage_off = l.cnt_off + (B + 3) / 4 * 4;
    l.stage_cnt_off = l.stage_off + B * l.nblk * kListChunks;
    l.total = l.stage_cnt_off + (B * l.nblk + 3) / 4 * 4;
    return l;
}

// Block (x, b) decides chunks 256x .. 256x + 255 of sequence b: chunk c is
// visible if some query row i < n_q sees one of its positions, one inside the
// filled prefix (for causal windows at or before L - n_q + i) whose mask is
// not -inf.  Warp w reads the 32 chunks from 256x + 32w on, one coalesced
// 128-byte row of the mask per chunk and query row (all 32 rows in flight at
// once), and ballots them into a word; the block lists its visible chunks in
// order in its region of the staging area and stores their count.  The last
// block of the sequence to finish (a ticket in the workspace's per-segment
// counters, which are zero between launches and which it puts back to zero)
// turns the regions' counts into offsets and copies every region, in order,
// into the sequence's list row, eight entries in flight per thread, and
// writes the count.
__global__ void __launch_bounds__(kListThreads)
mask_chunk_list(const __grid_constant__ Params p, int32_t *list, int32_t *cnt, int32_t *stage,
                int32_t *stage_cnt, int32_t *tickets, int64_t mls, int32_t nblk) {
    __shared__ int wsum[kListThreads / 32];
    __shared__ int offs[kListMaxBlocks + 1];
    __shared__ int last;
    const int b = blockIdx.y, x = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t raw = (int64_t)__ldg(p.kv_lengths + b);
    const int64_t L = clamp_len(raw, p.cap);
    if (x == 0 && tid == 0 && (raw < 0 || raw > p.cap)) atomicOr(p.status, kDevBadLength);
    const float *mrow = p.mask + (int64_t)b * p.ms[0];
    const int64_t c0 = (int64_t)x * kListChunks + warp * 32;
    uint32_t word = 0;
    if (c0 * 32 < L) {
        uint32_t vis = 0;   // bit k: this lane's position of chunk c0 + k is seen
        for (int i = 0; i < p.n_q; ++i) {
            // positions this row sees: 0 .. lim - 1
            const int64_t lim = p.causal ? L - p.n_q + i + 1 : L;
            const float *mr = mrow + (int64_t)i * p.ms[1];
            float m[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int64_t pos = 32 * (c0 + k) + lane;
                m[k] = pos < lim ? __ldg(mr + pos) : neg_inf();
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) vis |= (m[k] != neg_inf() ? 1u : 0u) << k;
        }
#pragma unroll
        for (int k = 0; k < 32; ++k)
            if (__ballot_sync(0xffffffffu, (vis >> k) & 1u)) word |= 1u << k;
    }
    if (lane == 0) wsum[warp] = __popc(word);
    __syncthreads();
    int off = 0, tot = 0;
#pragma unroll
    for (int w2 = 0; w2 < kListThreads / 32; ++w2) {
        off += w2 < warp ? wsum[w2] : 0;
        tot += wsum[w2];
    }
    const int64_t region = (int64_t)b * nblk + x;
    if ((word >> lane) & 1u)
        stage[region * kListChunks + off + __popc(word & ((1u << lane) - 1u))] = (int32_t)(c0 + lane);
    if (tid == 0) stage_cnt[region] = tot;
    __threadfence();
    __syncthreads();
    if (tid == 0) last = atomicAdd(tickets + b, 1) == nblk - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    // regions' counts -> exclusive offsets (a block-wide scan per 256 regions)
    int carry = 0;
    for (int r0 = 0; r0 < nblk; r0 += kListThreads) {
        const int r = r0 + tid;
        const int n = r < nblk ? __ldcg(stage_cnt + (int64_t)b * nblk + r) : 0;
        int inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        __syncthreads();   // the previous pass's reads of wsum are done
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        int before = carry, all = carry;
#pragma unroll
        for (int w2 = 0; w2 < kListThreads / 32; ++w2) {
            before += w2 < warp ? wsum[w2] : 0;
            all += wsum[w2];
        }
        if (r < nblk) offs[r] = before + inc - n;
        carry = all;
    }
    if (tid == 0) offs[nblk] = carry;
    __syncthreads();
    // entry e of region r -> list position offs[r] + e
    int32_t *dst = list + (int64_t)b * mls;
    const int32_t *src = stage + (int64_t)b * nblk * kListChunks;
    for (int r0 = 0; r0 < nblk; r0 += 8) {
        int32_t v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int r = r0 + u;
            v[u] = r < nblk && tid < offs[r + 1] - offs[r] ? __ldcg(src + (int64_t)r * kListChunks + tid) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int r = r0 + u;
            if (r < nblk && tid < offs[r + 1] - offs[r]) dst[offs[r] + tid] = v[u];
        }
    }
    if (tid == 0) {
        cnt[b] = carry;
        tickets[b] = 0;
    }
}

}  // namespace

int64_t tc_mask_list_ints(int64_t B, int64_t cap) {
    const ListLayout l = list_layout(B, cap);
    return B > 65535 || l.nblk > kListMaxBlocks ? 0 : l.total;
}

int launch_tc_masked_list(const Params &p, int G, cudaStream_t st) {
    const ListLayout l = list_layout(p.B, p.cap);
    if (p.B > 65535 || l.nblk > kListMaxBlocks) return -2;
    int32_t *base = const_cast<int32_t *>(p.mlist);
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    args.p.mcnt = base + l.cnt_off;
    args.p.mls = l.mls;
    // 32-row boxes (one chunk) and 128-row boxes (four consecutive chunks)
    if (!make_map(&args.tk, p.k, p.ks, p, 32) || !make_map(&args.tv, p.v, p.vs, p, 32) ||
        !make_map(&args.gk, p.k, p.ks, p) || !make_map(&args.gv, p.v, p.vs, p) ||
        !make_qmap(&args.tq, p))
        return -5;
    mask_chunk_list<<<dim3((unsigned)l.nblk, (unsigned)p.B), kListThreads, 0, st>>>(
        p, base, base + l.cnt_off, base + l.stage_off, base + l.stage_cnt_off, p.counters, l.mls,
        (int32_t)l.nblk);
    if (cudaGetLastError() != cudaSuccess) return -5;
    const int rows = p.rows;
    if (p.d == 128)
        return rows <= 16   ? launch_dn<128, 16, false, 16, false, false, false, false, 2>(args, G, st)
               : rows <= 32 ? launch_dn<128, 32, false, 32, false, false, false, false, 2>(args, G, st)
               : rows <= 48 ? launch_dn<128, 48, false, 48, false, false, false, false, 2>(args, G, st)
                            : launch_dn<128, 64, false, 64, false, false, false, false, 2>(args, G, st);
    return rows <= 16   ? launch_dn<256, 16, false, 16, false, false, false, false, 2>(args, G, st)
           : rows <= 32 ? launch_dn<256, 32, false, 32, false, false, false, false, 2>(args, G, st)
           : rows <= 48 ? launch_dn<256, 48, false, 48, false, false, false, false, 2>(args, G, st)
                        : launch_dn<256, 64, false, 64, false, false, false, false, 2>(args, G, st);
}

}  // namespace fd
