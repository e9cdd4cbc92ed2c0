// fd_tc_kernel.cuh -- the tensor-core (tcgen05) decode kernel template and
// its host-side helpers (tensor-map encoding, occupancy, launch), included
// by the translation units that instantiate it: fd_tc.cu (flat caches,
// index gather) and fd_tc_paged.cu (paged caches).
//
// Modes: the dense prefix (optionally causal) over flat or paged caches, and
// index gather; bf16 caches at head_dim 128 / 256 with up to 64 packed query
// rows, int8 caches at head_dim 128 / 256 with up to 32.
//
// Work split: balanced consecutive ranges of work units over one block per
// SM, where a segment is its tiles (128 positions) plus a few units for the
// fixed cost of a piece boundary (see Walk).  Roles inside a block
// (320 threads):
//   warp 8      TMA producer: loads each segment's packed Q rows (one box
//               per 64 columns) as soon as the previous piece's last QK has
//               read the buffer, and streams K and V tiles of the block's
//               range into a ring of shared-memory slots (4-D tensor maps,
//               128-byte swizzle), in the order the MMAs consume them.
//   warp 9      MMA issuer (one thread): S^T = K . Q^T   (M = 128 positions,
//               N = padded query rows, K = head_dim) into TMEM, then
//               O^T += V^T . P^T (M = 128 dims per chunk, N = rows,
//               K = 128 positions) into TMEM; completion via tcgen05.commit.
//               QK of tile t+1 is issued before PV of tile t.
//   warps 0-7   softmax and epilogue, two warpgroups that split the query
//               rows (bf16 caches).  Thread i of a group owns TMEM lane i =
//               cache position i of the tile (scores) and dim i of each
//               128-dim chunk (output).  Per tile: mask (length, causal
//               window), running row maxima refreshed when a score passes
//               them by 2^8 (column max over the 128 positions by warp
//               shuffles + shared memory), O rescaled in TMEM then,
//               P = 2^(s - m) written to shared memory in the MMA operand
//               layout (one bf16 plane, or hi + lo planes for fp32 outputs).
//               At the end of a segment piece it normalises and stores, or
//               hands a split partial to the in-launch combine (last block
//               to arrive merges; comfy-kitchen #239, "GQA decode").
//   int8 caches: warps 0-3 are the one softmax group and warps 4-7 widen the
//               int8 tiles the producer loads into fp16 slots and convert
//               each piece's Q to fp16, so the MMAs run on fp16 operands (P
//               is written in fp16 too); the per-position scales multiply
//               scores and P.
// Flat caches: the last tile of a segment is loaded right-aligned (ending at
// the length), so no row of the unused tail is ever read; positions the
// previous tile already covered are masked.  Paged caches (PG) and index
// gather (GA): tiles start at multiples of 128 and each producer lane fetches
// four rows per tile with tile::gather4 (rows past the length, or of a bad
// page or cell, are row -1 and read as zeros; the softmax masks them).  Every wait is bounded (2 s); a timeout sets
// FD_DEV_INTERNAL in the status word, records where it waited, and the block
// drains its copies and MMAs and exits.
#pragma once

#include <cuda.h>
#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <cuda_runtime.h>

#include "fd_device.cuh"
#include "fd_launch.h"
#include "fd_ptx.cuh"

namespace fd {

// ------------------------------------------------------ tensor-map encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Tensor maps are encoded on the host for every launch; a decode loop passes
// the same caches (and often the same q) each step, so the last encodings
// are kept, keyed by every argument that goes into one.
struct MapKey {
    const void *base;
    uint32_t dtype, rank, swizzle, pad;
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
};

inline EncodeTiledFn encode_fn();

inline CUresult encode_cached(CUtensorMap *m, CUtensorMapDataType dtype, cuuint32_t rank, void *base,
                       const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                       const cuuint32_t *estr, CUtensorMapSwizzle swizzle) {
    MapKey k;
    memset(&k, 0, sizeof k);
    k.base = base;
    k.dtype = (uint32_t)dtype;
    k.rank = rank;
    k.swizzle = (uint32_t)swizzle;
    for (cuuint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    constexpr int kEntries = 32;
    static std::mutex mu;
    static MapKey keys[kEntries];
    static CUtensorMap maps[kEntries];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (memcmp(&keys[i], &k, sizeof k) == 0) {
                *m = maps[i];
                return CUDA_SUCCESS;
            }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_SUPPORTED;
    const CUresult r = fn(m, dtype, rank, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lk(mu);
        keys[next] = k;
        maps[next] = *m;
        next = (next + 1) % kEntries;
        if (used < kEntries) ++used;
    }
    return r;
}

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

namespace {

constexpr int TT = 128;                 // cache positions per tile (MMA M)
constexpr int kMaxGroups = 2;           // softmax warpgroups (bf16 caches)
constexpr int kThreadsTC = 320;         // warps 0-7, producer, MMA issuer
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
// Bound on the waits that drain a block's own copies and MMAs before it
// exits (they always end); the other waits take Params::wait_ns.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kDevTimeout = 4;          // mirrors FD_DEV_INTERNAL
constexpr uint32_t kBarsBytes = 512;    // barrier block; the reduction scratch follows
// Scores (log2 units) may exceed a row's running maximum by this much before
// the maximum is refreshed and O rescaled; P is then at most 2^8, which fp32
// accumulators and the hi/lo bf16 split of P carry without loss.
constexpr float kRescaleSlack = 8.f;

struct TcArgs {   // CUtensorMap members carry their own alignment
    // (int8 caches: tk / tv map the int8 codes; gather and paged caches: 2-D
    // maps of cache rows)
    CUtensorMap tk;
    CUtensorMap tv;
    CUtensorMap tq;
    Params p;
    // gather: cache row (b, hk, pos) is row b*gs0 + hk*gs1 + pos*gs2 of tk / tv;
    // paged: pool row (page, hk, r) is row page*gs0 + hk*gs1 + r*gs2 of gk / gv;
    // masked prefix: gk / gv load 128-row boxes, tk / tv 32-row chunks
    int64_t gs0, gs1, gs2;
    // paged: tk / tv are 4-D maps of the pool (d, page_size, Hkv, num_pages)
    // with box (64, prow, 1, 1); a tile wholly inside the length is TT / prow
    // such boxes (prow = 0: every tile is gathered row by row)
    CUtensorMap gk;
    CUtensorMap gv;
    int32_t prow;
};

template <int D, int N, bool I8, int NV, bool GA = false>
struct Cfg {
    // bf16 caches: two softmax warpgroups split the rows (warps 0-7).  int8
    // caches: one softmax warpgroup (warps 0-3); warps 4-7 widen the int8
    // tiles to fp16 for the MMAs.
    static constexpr int GROUPS = I8 ? 1 : 2;
    static constexpr int SMT = 128 * GROUPS;     // softmax threads
    static constexpr int KB = D / 64;            // 128-byte boxes per cache row
    static constexpr int DC = D / 128;           // 128-dim chunks of O
    static constexpr uint32_t BOX = TT * 128;    // bytes of one box of a slot
    static constexpr uint32_t SLOT = KB * BOX;   // one K or V tile
    static constexpr uint32_t QB = N * 128;      // one 64-column box of Q or P
    static constexpr uint32_t QBYTES = KB * QB;
    static constexpr uint32_t PPLANE = 2 * QB;   // one bf16 plane of P (128 positions x N)
    static constexpr uint32_t PSTAGE = 2 * PPLANE;   // P = hi plane + lo plane
    // Query rows per softmax warpgroup.
    // Rows the softmax handles: NV (<= N, a multiple of 8) bounds the packed
    // rows; the MMAs still run N columns, and P rows NV..N-1 stay zero.
    static_assert(NV <= N && NV % 8 == 0, "valid-row bound");
    static constexpr int NH = NV / GROUPS;
    static_assert(NH % 8 == 0, "rows per group must be a multiple of 8");
    // Barriers and the reduction scratch come first, then 1024-byte aligned
    // operand buffers.  Scratch per group: [2 tiles][4 warps][NH] floats.
    static constexpr uint32_t RED_GROUP = 2 * 4 * NH;   // floats
    static constexpr uint32_t RED = GROUPS * RED_GROUP * 4;
    // Per-row element offsets into out for the current segment (int64), two
    // tables used by alternate pieces.
    static constexpr uint32_t OFF_TBL = kBarsBytes + RED;
    static constexpr uint32_t TBL = 2 * N * 8;
    static constexpr uint32_t MISC = ((OFF_TBL + TBL) + 1023) / 1024 * 1024;
    static constexpr uint32_t BUDGET = 232448;   // max dynamic shared memory per block
    // int8 caches: a ring of NR raw tiles (TT positions x D codes, as TMA
    // lands them) in front of the fp16 slots the MMAs read.
    static constexpr uint32_t RAW = I8 ? TT * D : 0;
    static constexpr int NR = I8 ? (D == 128 ? 3 : 2) : 0;
    static constexpr int NRX = I8 ? NR : 1;   // ring length for index arithmetic
    // Two P stages when that still leaves three K/V slots, else one.
    static constexpr int NS2 = (int)((BUDGET - MISC - QBYTES - 2 * PSTAGE - NR * RAW) / SLOT);
    static constexpr int PST = NS2 >= 3 ? 2 : 1;
    static constexpr int NS_RAW = (int)((BUDGET - MISC - QBYTES - PST * PSTAGE - NR * RAW) / SLOT);
    static constexpr int NS = NS_RAW > 8 ? 8 : NS_RAW;
    static_assert(NS >= 2, "need two K/V slots");
    static constexpr uint32_t OFF_SLOTS = MISC;
    static constexpr uint32_t OFF_Q = OFF_SLOTS + NS * SLOT;
    static constexpr uint32_t OFF_P = OFF_Q + QBYTES;
    static constexpr uint32_t OFF_RAW = OFF_P + PST * PSTAGE;
    static constexpr uint32_t SMEM = OFF_RAW + NR * RAW;
    // (the fused-append exit path declares a few bytes of static shared memory)
    static_assert(SMEM + 64 <= BUDGET, "shared memory budget");
    static constexpr uint32_t COLS = 2 * N + DC * N;
    static constexpr uint32_t TMEM_COLS = COLS <= 32 ? 32 : COLS <= 64 ? 64 : COLS <= 128 ? 128 : 256;
    // pieces per iteration of the last arriver's single-pass merge (head_dim 256)
    static constexpr int MERGE_UNROLL = (D == 256 && NV >= 32 && !I8) ? 1 : 2;
    // int8 caches: the MMAs take fp16 operands (codes widen to fp16 in two
    // instructions per pair, Q is converted once per piece, P is written in
    // fp16); bf16 caches: bf16 operands
    static constexpr uint32_t IDESC_QK = I8 ? ptx::idesc_f16(128, N, 0, 0) : ptx::idesc_bf16(128, N, 0, 0);
    static constexpr uint32_t IDESC_PV = I8 ? ptx::idesc_f16(128, N, 1, 1) : ptx::idesc_bf16(128, N, 1, 1);
    // Scores (log2 units) may exceed a row's running maximum by this much
    // before the maximum is refreshed, so P <= 2^SLACK: fp32 accumulators
    // and the hi/lo split of P (bf16, or fp16 for int8 caches, where P also
    // carries the position's v scale and must stay below the fp16 maximum)
    // carry it without loss.
    static constexpr float SLACK = I8 ? 4.f : kRescaleSlack;
    // P planes are MN-major (query rows contiguous per position) with 32-byte
    // swizzle: 16-row atoms of TT positions x 32 bytes.
    static constexpr uint32_t PATOM = TT * 32;
};

// ------------------------------------------------------------------ pieces
// The split is over work units: a non-empty segment s = b*Hkv + hk holds
// V = p.seg_units units that stand for the fixed cost of a piece boundary
// (epilogue, pipeline restart), then one unit per tile.  The block whose
// range crosses into a segment pays for the boundary with V fewer tiles; a
// range may start or end inside those V units, which map to no tile.
// A block's work is a run of consecutive non-empty segments.  The first one
// is found once per block by a warp scan over the sequence lengths; every
// later one is the next non-empty segment, so walking needs no division.
// Gather launches: segment s = (b*n_q + i)*Hkv + hk is one index list (all of
// length idx_len) seen by the g query heads of kv head hk.
struct Walk {
    int64_t s;        // segment
    int64_t first;    // unit index of the segment's first tile
    int64_t L;        // positions walked: the sequence length (gather: the list
                      // length; masked with a chunk list: 32 per listed chunk)
    int32_t ntiles;   // its tile count
    int32_t b, hk;
    int32_t i;        // gather: query row of the list (dense: 0)
};

__device__ __forceinline__ int32_t tiles_of(int64_t L) { return (int32_t)((L + TT - 1) / TT); }

// Positions a segment of sequence b walks: its length, or, for the masked
// prefix with a chunk list, 32 per listed chunk (tile t of the segment then
// holds list entries 4t .. 4t+3).  A count outside [0, ceil(cap / 32)] reads
// as that bound.
__device__ __forceinline__ int64_t walk_len(const Params &p, int b) {
    if (!p.mcnt) return seq_len(p, b);
    const int64_t n = (int64_t)__ldg(p.mcnt + b), nmax = (p.cap + 31) / 32;
    return 32 * (n < 0 ? 0 : n > nmax ? nmax : n);
}

// Units of a segment of n tiles.
__device__ __forceinline__ int64_t units_of(const Params &p, int64_t n) {
    return n > 0 ? n + p.seg_units : 0;
}

// Total work units of the launch (one warp; every lane gets the value).
__device__ __forceinline__ int64_t total_units_tc(const Params &p) {
    if (p.mode == kGather) return p.nseg * units_of(p, tiles_of(p.idx_len));
    const int lane = threadIdx.x & 31;
    int64_t acc = 0;
    for (int b = lane; b < p.B; b += 32) acc += units_of(p, tiles_of(walk_len(p, b)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc * p.Hkv;
}

// The segment holding work unit t (one warp; false if t is past the end).
__device__ __noinline__ bool first_piece_warp(const Params &p, int64_t t, Walk *w) {
    if (p.mode == kGather) {   // equal segments: closed form
        const int64_t n = tiles_of(p.idx_len), u = units_of(p, n);
        if (u == 0 || t >= p.nseg * u) return false;
        const int64_t s = t / u, bi = s / p.Hkv;
        w->s = s;
        w->hk = (int)(s % p.Hkv);
        w->b = (int)(bi / p.n_q);
        w->i = (int)(bi % p.n_q);
        w->first = s * u + p.seg_units;
        w->ntiles = (int32_t)n;
        w->L = p.idx_len;
        return true;
    }
    const int lane = threadIdx.x & 31;
    int64_t base = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        const int64_t L = b < p.B ? walk_len(p, b) : 0;
        const int64_t n = tiles_of(L), u = units_of(p, n);
        const int64_t wt = (int64_t)p.Hkv * u;
        int64_t incl = wt;   // inclusive scan over the 32 lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        const int64_t excl = incl - wt;
        const unsigned m = __ballot_sync(0xffffffffu, wt > 0 && t >= base + excl && t < base + incl);
        if (m) {
            const int src = __ffs(m) - 1;
            const int64_t e = __shfl_sync(0xffffffffu, excl, src);
            const int64_t nb = __shfl_sync(0xffffffffu, n, src);
            const int64_t ub = __shfl_sync(0xffffffffu, u, src);
            const int64_t Lb = __shfl_sync(0xffffffffu, L, src);
            const int hk = (int)((t - base - e) / ub);
            w->b = b0 + src;
            w->hk = hk;
            w->i = 0;
            w->s = (int64_t)w->b * p.Hkv + hk;
            w->first = base + e + (int64_t)hk * ub + p.seg_units;
            w->ntiles = (int32_t)nb;
            w->L = Lb;
            return true;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    return false;
}

// Advance to the next segment with at least one tile (false past the end).
__device__ __forceinline__ bool next_piece(const Params &p, Walk &w) {
    w.first += w.ntiles;
    if (p.mode == kGather) {
        if (w.s + 1 >= p.nseg) return false;
        ++w.s;
        if (++w.hk == p.Hkv) {
            w.hk = 0;
            if (++w.i == p.n_q) {
                w.i = 0;
                ++w.b;
            }
        }
        w.first += p.seg_units;
        return true;
    }
    do {
        if (w.s + 1 >= p.nseg) return false;
        ++w.s;
        if (++w.hk == p.Hkv) {
            w.hk = 0;
            ++w.b;
            w.L = walk_len(p, w.b);
            w.ntiles = tiles_of(w.L);
        }
    } while (w.ntiles == 0);
    w.first += p.seg_units;
    return true;
}

struct Bars {   // at the start of shared memory; the reduction scratch follows at kBarsBytes
    uint64_t slot_full[8], slot_empty[8];
    uint64_t s_full[2], s_free[2], p_full[2], p_free[2];
    uint64_t q_full, q_free, o_done, o_free, exit_mma, sm_bar;
    uint64_t q_conv;          // int8 caches: Q converted to fp16 (the widening threads)
    uint64_t wg_bar[kMaxGroups];
    union {
        struct {
            uint64_t raw_full[6], raw_empty[6];   // int8 caches: raw tile ring
        };
        Walk walk_last;   // shared merges (bf16 caches): the last piece worked on
    };
    uint32_t tmem_base;
    int abort_flag;
    int last_flag;
    int pad;
    int64_t total;
    int vote[kMaxGroups][2][4];
    int64_t t_begin, t_end;   // the block's range of work units
    Walk walk;                // its first piece
    int has_work;
};

// Ring fill index of the K and V tiles of tile number tc in a piece whose
// first and last tiles are pa and pb, for the fill order K(pa), K(pa+1),
// V(pa), K(pa+2), V(pa+1), ..., V(pb).
__device__ __forceinline__ uint32_t k_fill(uint32_t tc, uint32_t pa) {
    return tc == pa ? 2 * tc : 2 * tc - 1;
}
__device__ __forceinline__ uint32_t v_fill(uint32_t tc, uint32_t pb) {
    return tc == pb ? 2 * tc + 1 : 2 * tc + 2;
}

// First cache position loaded for tile tt of a segment of length L: tiles
// start at tt * TT, except the last, which is right-aligned to end at L (its
// start may be negative, where TMA fills zeros), so no position past the
// filled prefix is ever loaded.
__device__ __forceinline__ int64_t tile_start(int64_t tt, int64_t L) {
    const int64_t y0 = tt * TT;
    return y0 + TT > L ? L - TT : y0;
}

static_assert(sizeof(Bars) <= kBarsBytes, "barrier block overlaps the reduction scratch");

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Two int8 codes (bytes k and k+1 of u = w ^ 0x80808080, i.e. code + 128)
// -> two fp16 holding the same integers, exactly: each byte becomes the low
// mantissa byte of the half 0x64XX = 1024 + byte, from which 1152 is
// subtracted exactly (fp16 holds integers of magnitude <= 2048 exactly).
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t u, int k) {
    const uint32_t h = __byte_perm(u, 0x64646464u, k == 0 ? 0x4140 : 0x4342);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

// Two floats -> two fp16 (round to nearest even, saturating at +-65504).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float f16lo(uint32_t w) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(w));
    return f;
}
__device__ __forceinline__ float f16hi(uint32_t w) {
    float f;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(w));
    return f;
}

__device__ __forceinline__ int ld_acquire(const int32_t *ptr) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ void set_abort(Bars *bs, const Params &p) {
    bs->abort_flag = 1;
    atomicOr(p.status, kDevTimeout);
}

// A wait that gives up records where (read back by fd_get_device_diagnostics):
// status[1..3] = site, tile counter and piece index of the first one in the
// launch; status[4 + 3r .. 6 + 3r] the same for the first failing wait of
// role r (0 producer, 1 MMA issuer, 2 softmax), so a stall shows what every
// role was blocked on when the block gave up.
__device__ __forceinline__ void note_timeout(Bars *bs, const Params &p, int site,
                                             uint32_t tile, int piece) {
    if (!bs->abort_flag && atomicCAS(p.status + 1, 0, site) == 0) {
        p.status[2] = (int)tile;
        p.status[3] = piece;
    }
    const int role = (site == 1 || site == 8) ? 0 : (site <= 7 ? 1 : 2);
    if (atomicCAS(p.status + 4 + 3 * role, 0, site) == 0) {
        p.status[5 + 3 * role] = (int)tile;
        p.status[6 + 3 * role] = piece;
    }
    set_abort(bs, p);
}

// One block's share of the merge of split segment sw.s (blocks c0 .. c1 hold
// its pieces) in a cooperative launch: wait until every piece has arrived,
// merge units [share*U/P, (share+1)*U/P) of the rows x (D/4) float4 units from
// the pieces' workspace slots (running maximum per row, pieces in order),
// store them, and count the share done (the last one resets the counter).
// A share of few units splits each unit's pieces over G threads (pieces
// g, g + G, ...), so G times as many loads are in flight, and merges the G
// partials through shared memory (scr: the block's free operand slots).
// Kept out of line so that its registers do not weigh on the tile loop.
template <int D, bool GA, int SMT>
__device__ __noinline__ bool share_merge_segment(const Params &p, Bars *bs, float *scr, Walk sw, int c0,
                                                 int c1, int c, int tid, uint32_t &sm_ctr, int k,
                                                 int piece) {
    volatile int *abort_flag = &bs->abort_flag;
    auto sm_sync = [&]() -> bool {
        ptx::mbar_arrive(&bs->sm_bar);
        if (ptx::mbar_wait(&bs->sm_bar, (sm_ctr++) & 1, abort_flag, p.wait_ns)) return true;
        note_timeout(bs, p, 14, 0, piece);
        return false;
    };
    const int64_t sg = sw.s;
    const int P = c1 - c0 + 1, share = c - c0;
    const int kSoftmaxThreads = SMT;
    bool ok;
    if (tid == 0) {
        const uint64_t t0 = ptx::globaltimer_ns();
        for (uint32_t n = 0; ld_acquire(p.counters + sg) < P; ++n) {
            __nanosleep(64);
            if ((n & 63) == 63 &&
                (*abort_flag || ptx::globaltimer_ns() - t0 > p.wait_ns)) {
                note_timeout(bs, p, 15, (uint32_t)k, piece);
                break;
            }
        }
    }
    ok = sm_sync() && !*abort_flag;
    if (!ok) return false;
    __threadfence();
    const int rows = p.rows;
    constexpr int UPR = D / 4;                    // float4 units per row
    const int64_t U = (int64_t)rows * UPR;
    const int64_t u0 = U * share / P, u1 = U * (share + 1) / P;
    const int nu = (int)(u1 - u0);
    // One step of the running-maximum merge: fold partial (mv, lv, v) into
    // (M, Ls, acc).  (Explicit roundings: the same arithmetic as the last
    // arriver's single-pass merge.)
    auto fold = [](float &M, float &Ls, float4 &acc, float mv, float lv, float4 v) {
        const float mn = fmaxf(M, mv);
        const float mu = mn == neg_inf() ? 0.f : mn;
        const float a = fast_exp2(M - mu), wv = fast_exp2(mv - mu);
        M = mn;
        Ls = __fmaf_rn(wv, lv, Ls * a);
        acc.x = __fmaf_rn(wv, v.x, acc.x * a);
        acc.y = __fmaf_rn(wv, v.y, acc.y * a);
        acc.z = __fmaf_rn(wv, v.z, acc.z * a);
        acc.w = __fmaf_rn(wv, v.w, acc.w * a);
    };
    // Unit u's pieces c0 + g, c0 + g + G, ... in order.
    auto merge_pieces = [&](int64_t u, int g, int G, float &M, float &Ls, float4 &acc) {
        const int r = (int)(u / UPR), dq = (int)(u % UPR) * 4;
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
        M = neg_inf();
        Ls = 0.f;
#pragma unroll 4
        for (int c2 = c0 + g; c2 <= c1; c2 += G) {
            const float *sl = slot_ptr(p, sg, c2);
            const float mv = __ldcg(sl + rows * D + r), lv = __ldcg(sl + rows * D + rows + r);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(sl + r * D + dq));
            fold(M, Ls, acc, mv, lv, v);
        }
    };
    auto store = [&](int64_t u, float Ls, float4 acc) {
        const int r = (int)(u / UPR), dq = (int)(u % UPR) * 4;
        const int qi = GA ? sw.i : r % p.n_q, h = sw.hk * p.g + (GA ? r : r / p.n_q);
        const int64_t off = (int64_t)sw.b * p.os[0] + (int64_t)qi * p.os[1] +
                            (int64_t)h * p.os[2] + dq;
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const float o4[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (p.out_f32)
                reinterpret_cast<float *>(p.out)[off + e] = o4[e];
            else
                reinterpret_cast<uint16_t *>(p.out)[off + e] = bf16_bits(o4[e]);
        }
    };
    const int G = (nu > 0 && 2 * nu <= kSoftmaxThreads) ? min(P, kSoftmaxThreads / nu) : 1;
    if (G >= 2) {
        // thread tid = g * nu + i: group g of unit u0 + i
        float4 *s4 = reinterpret_cast<float4 *>(scr);
        float *sm = scr + 4 * kSoftmaxThreads, *sl = sm + kSoftmaxThreads;
        if (tid < G * nu) {
            const int g = tid / nu;
            float M, Ls;
            float4 acc;
            merge_pieces(u0 + (tid - g * nu), g, G, M, Ls, acc);
            s4[tid] = acc;
            sm[tid] = M;
            sl[tid] = Ls;
        }
        ok = sm_sync();
        if (!ok) return false;
        if (tid < nu) {
            float M = neg_inf(), Ls = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int g = 0; g < G; ++g) fold(M, Ls, acc, sm[g * nu + tid], sl[g * nu + tid], s4[g * nu + tid]);
            store(u0 + tid, Ls, acc);
        }
    } else {
        for (int64_t u = u0 + tid; u < u1; u += kSoftmaxThreads) {
            float M, Ls;
            float4 acc;
            merge_pieces(u, 0, 1, M, Ls, acc);
            store(u, Ls, acc);
        }
    }
    ok = sm_sync();
    if (!ok) return false;
    if (tid == 0 && atomicAdd(p.counters + sg, 1) == 2 * P - 1) p.counters[sg] = 0;
    return true;
}

// The last arriver's merge of split segment s (pieces in blocks c_first ..
// c_last): rows cb0 .. r1w-1 (one softmax group's), thread wt of the group.
template <int D, int NH, int MU>
__device__ __forceinline__ void merge_split_rows(const Params &p, int64_t s, int c_first, int c_last,
                                                 int cb0, int r1w, int wt, const int64_t *ooff) {
    const int rows = p.rows;
    // Merge the pieces' partials.  head_dim 128 (launches
    // that often split a segment many ways): two passes per
    // row, the maximum M over the pieces, then the weighted
    // sums Ls and acc (weights 2^(m - M)), neither carrying a
    // dependence from one piece's loads to the next, so many
    // pieces' loads are in flight together.  head_dim 256:
    // one pass with a running maximum (the shared merge's
    // fold of one partial; a smaller loop body, which
    // runs once from cold instruction caches).  Thread -> 4
    // consecutive dims of rows cb0 + rg + RG*k; row indices
    // are clamped into range (weight 0 beyond) so every load
    // is unconditional.
    constexpr int TPR = D / 4, RG = 128 / TPR, RPT = NH / RG;
    constexpr int CH = RPT < 8 ? RPT : 8;
    const int dq = (wt % TPR) * 4, rg = wt / TPR;
#pragma unroll 1
    for (int k0 = 0; k0 < RPT && cb0 + rg + RG * k0 < r1w; k0 += CH) {
        float4 acc[CH];
        float M[CH], Ls[CH];
        int rr[CH];
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int r = cb0 + rg + RG * (k0 + k);
            rr[k] = r < r1w ? r : r1w - 1;
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            M[k] = neg_inf();
            Ls[k] = 0.f;
        }
        if (D == 128) {
#pragma unroll 8
            for (int c2 = c_first; c2 <= c_last; ++c2) {
                const float *sl = slot_ptr(p, s, c2);
#pragma unroll
                for (int k = 0; k < CH; ++k) M[k] = fmaxf(M[k], __ldcg(sl + rows * D + rr[k]));
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) M[k] = M[k] == neg_inf() ? 0.f : M[k];
#pragma unroll 4
            for (int c2 = c_first; c2 <= c_last; ++c2) {
                const float *sl = slot_ptr(p, s, c2);
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const float mv = __ldcg(sl + rows * D + rr[k]);
                    const float lv = __ldcg(sl + rows * D + rows + rr[k]);
                    const float4 v =
                        __ldcg(reinterpret_cast<const float4 *>(sl + rr[k] * D + dq));
                    const float w = fast_exp2(mv - M[k]);
                    Ls[k] = __fmaf_rn(w, lv, Ls[k]);
                    acc[k].x = __fmaf_rn(w, v.x, acc[k].x);
                    acc[k].y = __fmaf_rn(w, v.y, acc[k].y);
                    acc[k].z = __fmaf_rn(w, v.z, acc[k].z);
                    acc[k].w = __fmaf_rn(w, v.w, acc[k].w);
                }
            }
        } else {
#pragma unroll(MU)
            for (int c2 = c_first; c2 <= c_last; ++c2) {
                const float *sl = slot_ptr(p, s, c2);
#pragma unroll
                for (int k = 0; k < CH; ++k) {
                    const float mv = __ldcg(sl + rows * D + rr[k]);
                    const float lv = __ldcg(sl + rows * D + rows + rr[k]);
                    const float4 v =
                        __ldcg(reinterpret_cast<const float4 *>(sl + rr[k] * D + dq));
                    const float mn = fmaxf(M[k], mv);
                    const float mu = mn == neg_inf() ? 0.f : mn;
                    const float a = fast_exp2(M[k] - mu), w = fast_exp2(mv - mu);
                    // (explicit roundings: the shared merge folds a
                    // partial with the same operations)
                    M[k] = mn;
                    Ls[k] = __fmaf_rn(w, lv, Ls[k] * a);
                    acc[k].x = __fmaf_rn(w, v.x, acc[k].x * a);
                    acc[k].y = __fmaf_rn(w, v.y, acc[k].y * a);
                    acc[k].z = __fmaf_rn(w, v.z, acc[k].z * a);
                    acc[k].w = __fmaf_rn(w, v.w, acc[k].w * a);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < CH; ++k) {
            const int r = cb0 + rg + RG * (k0 + k);
            if (r < r1w) {
                const int64_t off = ooff[r] + dq;
                const float inv = Ls[k] > 0.f ? 1.f / Ls[k] : 0.f;
                const float o4[4] = {acc[k].x * inv, acc[k].y * inv, acc[k].z * inv,
                                     acc[k].w * inv};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (p.out_f32)
                        reinterpret_cast<float *>(p.out)[off + e] = o4[e];
                    else
                        reinterpret_cast<uint16_t *>(p.out)[off + e] = bf16_bits(o4[e]);
                }
            }
        }
    }
}

// The same, out of line: the flat int8 kernels with up to 8 rows (one
// softmax group, widening warps beside it) run measurably faster with the
// merge's registers and code outside the softmax loop (the int8 workload
// 313.6 -> 296.5 us); every other instantiation is faster with it inline.
template <int D, int NH, int MU>
__device__ __noinline__ void merge_split_rows_ool(const Params &p, int64_t s, int c_first, int c_last,
                                                  int cb0, int r1w, int wt, const int64_t *ooff) {
    merge_split_rows<D, NH, MU>(p, s, c_first, c_last, cb0, r1w, wt, ooff);
}

// Gather with cluster merges: this block's share of the merge of its
// cluster's list.  The partial of block k (O[rows][D], m[rows], l[rows],
// fp32) sits at shared address `part` of block k; thread tid of this block
// (rank `rank`) merges float4 units rank * U / cl + tid, + 320, ... below
// (rank + 1) * U / cl of the U = rows * D / 4, reading every block's partial
// through distributed shared memory, and stores the normalised outputs.
template <int D>
__device__ __noinline__ void cluster_merge(const Params &p, uint32_t part, int tid) {
    const int cs = p.cl, rank = (int)ptx::cluster_ctarank(), rows = p.rows;
    const int64_t sg = ptx::cluster_id_x();
    if (sg >= p.nseg) return;
    const int64_t bi = sg / p.Hkv;
    const int hk = (int)(sg % p.Hkv), b = (int)(bi / p.n_q), i = (int)(bi % p.n_q);
    constexpr int UPR = D / 4;
    const int U = rows * UPR;
    const int u0 = (int)((int64_t)U * rank / cs), u1 = (int)((int64_t)U * (rank + 1) / cs);
    for (int u = u0 + tid; u < u1; u += kThreadsTC) {
        const int r = u / UPR, dq = (u % UPR) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float M = neg_inf(), Ls = 0.f;
        for (int k = 0; k < cs; ++k) {
            const uint32_t pk = ptx::map_cluster(part, (uint32_t)k);
            const float mv = ptx::ld_cluster_f32(pk + (uint32_t)(rows * D + r) * 4);
            if (mv == neg_inf()) continue;   // nothing seen (a block without tiles holds no O)
            const float lv = ptx::ld_cluster_f32(pk + (uint32_t)(rows * D + rows + r) * 4);
            const float4 v = ptx::ld_cluster_f32x4(pk + (uint32_t)(r * D + dq) * 4);
            const float mn = fmaxf(M, mv);
            const float mu = mn == neg_inf() ? 0.f : mn;
            const float a = fast_exp2(M - mu), w = fast_exp2(mv - mu);
            M = mn;
            Ls = __fmaf_rn(w, lv, Ls * a);
            acc.x = __fmaf_rn(w, v.x, acc.x * a);
            acc.y = __fmaf_rn(w, v.y, acc.y * a);
            acc.z = __fmaf_rn(w, v.z, acc.z * a);
            acc.w = __fmaf_rn(w, v.w, acc.w * a);
        }
        const int64_t off = (int64_t)b * p.os[0] + (int64_t)i * p.os[1] +
                            (int64_t)(hk * p.g + r) * p.os[2] + dq;
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const float o4[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (p.out_f32)
                reinterpret_cast<float *>(p.out)[off + e] = o4[e];
            else
                reinterpret_cast<uint16_t *>(p.out)[off + e] = bf16_bits(o4[e]);
        }
    }
}

// Fused append: this block's share of the new rows, copied into the caches
// (16-byte chunks spread over every thread of the grid).
__device__ __noinline__ void append_rows(const Params &p) {
    const int cpr = p.d / 8;
    const int64_t per = (int64_t)p.B * p.Hkv * p.n_new * cpr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < 2 * per; e += stride) {
        const int which = e >= per;
        int64_t r = which ? e - per : e;
        const int cc = (int)(r % cpr);
        r /= cpr;
        const int i = (int)(r % p.n_new);
        r /= p.n_new;
        const int hk = (int)(r % p.Hkv);
        const int b = (int)(r / p.Hkv);
        const int64_t pos = append_base(p, b) + i;
        if (pos >= p.cap) continue;
        const int64_t *ns = which ? p.vns : p.kns;
        const int64_t *cs = which ? p.vs : p.ks;
        const uint16_t *src = (which ? p.v_new : p.k_new) + (int64_t)b * ns[0] + (int64_t)i * ns[1] +
                              (int64_t)hk * ns[2] + cc * 8;
        uint16_t *dst = const_cast<uint16_t *>(static_cast<const uint16_t *>(which ? p.v : p.k)) +
                        (int64_t)b * cs[0] + (int64_t)hk * cs[1] + pos * cs[2] + cc * 8;
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    }
}

// Fused append: every block of the (cooperative, all blocks resident)
// launch counts itself in once its share of the new rows is written ...
__device__ __noinline__ void append_arrive(const Params &p) {
    ptx::fence_proxy_async_global();
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(p.grid, 1);
}

// ... and the producer waits for every block's count before its first cache
// read, so no TMA load of a tile holding new positions starts before they
// are in the caches (set-up overlaps the wait).  Bounded; giving up sets
// FD_DEV_INTERNAL and the launch's output is not valid.
__device__ __noinline__ void append_wait(const Params &p) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t n = 0; ld_acquire(p.grid) < (int)gridDim.x; ++n) {
        __nanosleep(32);
        if ((n & 63) == 63 && ptx::globaltimer_ns() - t0 > p.wait_ns) {
            atomicOr(p.status, kDevTimeout);
            break;
        }
    }
}

// Bounded mbarrier wait.  Kernels whose hot loops crowd the instruction
// caches keep only the first test inline and call the waiting loop: the int8
// kernels in the producer, MMA and widening roles (few live registers
// there), and in the softmax too where it has registers to spare (up to 8
// rows).
template <bool OOL>
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         uint64_t limit_ns) {
    if (OOL) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        return ptx::mbar_wait_slow(bar, parity, abort, limit_ns);
    }
    return ptx::mbar_wait(bar, parity, abort, limit_ns);
}

template <int D, int N, bool I8, int NV, bool GA, bool SH, bool PG, bool AP, int MK, bool CL>
__global__ void __launch_bounds__(kThreadsTC, 1) tc_kernel(const __grid_constant__ TcArgs a) {
    static_assert(!(GA && PG), "gather and paged loads are separate modes");
    static_assert(!AP || (!I8 && !GA && !PG), "fused append: flat bf16 caches");
    static_assert(!MK || (!I8 && !GA && !PG && !AP && !SH), "masked prefix: flat bf16 caches");
    // masked prefix: MK = 1 finds each tile's visible chunks in place, MK = 2
    // walks the chunk list of the pass before the launch
    static_assert(MK >= 0 && MK <= 2, "masked mode");
    static_assert(!CL || (GA && !I8 && !SH && !PG && !AP && !MK), "cluster merges: bf16 gather");
    constexpr bool MP = MK == 1, ML = MK == 2;
    using C = Cfg<D, N, I8, NV, GA>;
    constexpr int kSoftmaxThreads = C::SMT;
    const Params &p = a.p;
    extern __shared__ __align__(1024) unsigned char smem[];
    const uint32_t smem_base = ptx::smem_u32(smem);
    Bars *bs = reinterpret_cast<Bars *>(smem);
    float *red = reinterpret_cast<float *>(smem + kBarsBytes);   // per group [2][4][NH]
    // Row tables: element offset of packed row r in out, one table per piece
    // parity (a group may start the next piece while a lagging warp of it
    // still stores the previous one).
    int64_t *otbl = reinterpret_cast<int64_t *>(smem + C::OFF_TBL);
    volatile int *abort_flag = &bs->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    // The swizzled operand layouts need 1024-byte aligned buffers; the
    // dynamic shared window starts aligned, and a block that finds otherwise
    // reports it instead of computing.
    // Fused append: the new rows go into the caches before any tile is read
    // (the producer waits for every block's rows before its first load).
    if (AP) {
        append_rows(p);
        append_arrive(p);
    }
    if (smem_base & 1023u) {
        if (tid == 0) atomicOr(p.status, kDevTimeout);
        if (AP) append_exit(p);
        if (CL) {   // the cluster's blocks meet twice before they leave
            ptx::cluster_sync();
            ptx::cluster_sync();
        }
        return;
    }

    // Segments with nothing to attend still need their output rows zeroed.
    for (int64_t s = c; s < p.nseg; s += G)
        if ((GA ? tiles_of(p.idx_len) : tiles_of(walk_len(p, (int)(s / p.Hkv)))) == 0)
            zero_segment(p, s);
    // The producer warp finds the block's tile range and first piece while
    // the others set up barriers and TMEM.
    if (warp == kProducerWarp) {
        const int64_t tot = CL ? tiles_of(p.idx_len) : total_units_tc(p);
        Walk w{};
        int64_t tb = 0, te = 0;
        bool has = false;
        if (CL) {
            // cluster of p.cl blocks per list: block `rank` takes tiles
            // [rank * n / cl, (rank + 1) * n / cl) of list `cluster id`
            const int64_t sg = ptx::cluster_id_x(), rank = ptx::cluster_ctarank(), bi = sg / p.Hkv;
            w.s = sg;
            w.hk = (int)(sg % p.Hkv);
            w.b = (int)(bi / p.n_q);
            w.i = (int)(bi % p.n_q);
            w.first = 0;
            w.ntiles = (int32_t)tot;
            w.L = p.idx_len;
            tb = rank * tot / p.cl;
            te = (rank + 1) * tot / p.cl;
            has = sg < p.nseg && tb < te;
        } else if (tot > 0) {
            const int32_t Gw = working_blocks(tot, G);
            if (c < Gw) {
                const Split sp{tot, Gw};
                tb = sp.start(c);
                te = sp.start(c + 1);
                has = tb < te && first_piece_warp(p, tb, &w) && w.first < te;
            }
        }
        if (lane == 0) {
            bs->total = tot;
            bs->t_begin = tb;
            bs->t_end = te;
            bs->walk = w;
            bs->has_work = has;
        }
    }
    if (tid == 0) {
        // K/V slots are filled by TMA (one arrival plus bytes) or, for int8
        // caches, by the 128 widening threads.
        for (int i = 0; i < C::NS; ++i) {
            ptx::mbar_init(&bs->slot_full[i], I8 ? 128 : 1);
            ptx::mbar_init(&bs->slot_empty[i], 1);
        }
        for (int i = 0; i < C::NR; ++i) {
            ptx::mbar_init(&bs->raw_full[i], 1);
            ptx::mbar_init(&bs->raw_empty[i], 128);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&bs->s_full[i], 1);
            ptx::mbar_init(&bs->s_free[i], kSoftmaxThreads);
            ptx::mbar_init(&bs->p_full[i], kSoftmaxThreads);
            ptx::mbar_init(&bs->p_free[i], 1);
        }
        ptx::mbar_init(&bs->q_full, 1);
        ptx::mbar_init(&bs->q_conv, 128);
        ptx::mbar_init(&bs->q_free, 1);
        ptx::mbar_init(&bs->o_done, 1);
        ptx::mbar_init(&bs->o_free, kSoftmaxThreads);
        ptx::mbar_init(&bs->exit_mma, 1);
        ptx::mbar_init(&bs->sm_bar, kSoftmaxThreads);
        for (int g = 0; g < C::GROUPS; ++g) ptx::mbar_init(&bs->wg_bar[g], 128);
        bs->abort_flag = 0;
        ptx::mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(&bs->tmem_base, C::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        ptx::prefetch_tmap(&a.tq);
        ptx::prefetch_tmap(&a.tk);
        ptx::prefetch_tmap(&a.tv);
        if (PG || MK) {
            ptx::prefetch_tmap(&a.gk);
            ptx::prefetch_tmap(&a.gv);
        }
    }
    // Masked prefix: the K / V slots start as zeros (a hidden tile is never
    // loaded and leaves the slot as it was, which must be finite).
    if (MK && tid < kSoftmaxThreads) {
        for (uint32_t e = tid; e < C::NS * C::SLOT / 16; e += kSoftmaxThreads)
            *reinterpret_cast<uint4 *>(smem + C::OFF_SLOTS + e * 16) = make_uint4(0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    // P rows NV..N-1 are never written: zero them once.
    if (NV < N && tid < kSoftmaxThreads) {
        for (uint32_t e = tid; e < C::PST * C::PSTAGE / 16; e += kSoftmaxThreads)
            *reinterpret_cast<uint4 *>(smem + C::OFF_P + e * 16) = make_uint4(0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    // Padding rows (p.rows .. N-1) of the Q operand stay zero: the Q copies
    // write only the segment's rows.
    if (tid < kSoftmaxThreads && p.rows < N) {
        const int per = (N - p.rows) * 8;    // 16-byte chunks per 64-column box
        for (int e = tid; e < C::KB * per; e += kSoftmaxThreads) {
            const int cb = e / per, rem = e - cb * per;
            *reinterpret_cast<uint4 *>(smem + C::OFF_Q + cb * C::QB + (p.rows + rem / 8) * 128 +
                                       (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bs->tmem_base;
    const bool has_work = bs->has_work != 0;
    const int64_t t_begin = bs->t_begin, t_end = bs->t_end;
    const Split sp{bs->total, has_work ? working_blocks(bs->total, G) : 1};
    // Shared merges (SH instantiations, cooperative launch): every block of a
    // split segment merges a share of it, which pays off when blocks stream
    // few tiles each (the last arriver's merge of many small pieces would be
    // the launch's tail); with longer ranges the last arriver merges.
    const bool share_merge = SH && p.coop && sp.total <= 4 * (int64_t)sp.G;
    const uint32_t q_addr = smem_base + C::OFF_Q;
    const uint32_t p_addr = smem_base + C::OFF_P;

    if (!has_work) {
        // nothing to stream: straight to the exit
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------ TMA producer
        if (AP) {
            if (lane == 0) append_wait(p);
            __syncwarp();
            ptx::fence_proxy_async_global();
        }
        uint32_t issued = 0;
        bool ok = true;
        int piece = 0;
        Walk w = bs->walk;
        int64_t t = max(t_begin, w.first);
        while (ok) {
            const int64_t piece_end = min(t_end, w.first + w.ntiles);
            const int b = w.b, hk = w.hk;
            // flat int8 caches served in parts of a kv head's query heads:
            // the caches' kv head of part hk
            const int hkc = (I8 && !GA && !PG) && p.kvdiv > 1 ? hk / p.kvdiv : hk;
            const int64_t L = w.L;
            // The segment's Q rows, once the previous piece's last QK has read
            // the buffer: one box per 64 columns covering query indices
            // 0..n_q-1 of query heads hk*g .. hk*g+g-1, which lands row
            // r = (head offset) * n_q + (query index), K-major with the
            // 128-byte swizzle the QK descriptors expect.
            if (lane == 0) {
                if (piece > 0) {
                    ok = bar_wait<I8>(&bs->q_free, (piece - 1) & 1, abort_flag, p.wait_ns);
                    if (!ok) note_timeout(bs, p, 8, issued, piece);
                }
                if (ok) {
                    // (gather: the list's one query row, box (64, 1, g, 1))
                    ptx::mbar_arrive_expect_tx(&bs->q_full, (uint32_t)(C::KB * p.rows * 128));
#pragma unroll
                    for (int cb = 0; cb < C::KB; ++cb)
                        ptx::tma_load_4d(smem + C::OFF_Q + cb * C::QB, &a.tq, &bs->q_full, cb * 64,
                                         GA ? w.i : 0, hk * p.g, b);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            // Fill order = MMA consumption order: K(a); then K(t+1), V(t) for
            // t = a .. b-1; then V(b) (a, b: first and last tile of the piece).
            // The ring is then a plain FIFO, and each K tile is requested one
            // tile period before its QK needs it.
            const int64_t n_in = piece_end - t, tt0 = t - w.first;
            // gather: lane l fetches positions 4l .. 4l+3 of each tile, rows of
            // the 2-D cache maps (-1, read as zeros, for padding, cells past the
            // list or out of range); the next K tile's rows are read ahead.
            // paged: the same, with the rows of positions 4l .. 4l+3 found
            // through the block table (-1 past the length or for a bad page),
            // for the segment's partial last tile only; a tile wholly inside
            // the length is read with tiled box loads, one per run of prow
            // rows on one page: lane s < TT / prow holds run s's page (-1 for
            // a bad entry, which reads as zeros) and first row.
            const int32_t *ilist = GA ? p.idx + ((int64_t)b * p.n_q + w.i) * p.idx_len : nullptr;
            const int64_t segrow = GA ? (int64_t)b * a.gs0 + (int64_t)hk * a.gs1 : (int64_t)hk * a.gs1;
            int yk[4] = {-1, -1, -1, -1}, yv0[4] = {-1, -1, -1, -1}, yv1[4] = {-1, -1, -1, -1};
            auto list_rows = [&](int64_t tile, int *y) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int64_t pos = tile * TT + 4 * lane + r;
                    y[r] = -1;
                    if (GA && pos < p.idx_len) {
                        const int x = __ldg(ilist + pos);
                        if (x >= 0 && x < p.cap) y[r] = (int)(segrow + (int64_t)x * a.gs2);
                    }
                    if (PG && pos < L) {
                        const int32_t pg = page_of(p, b, (int32_t)pos);
                        if (pg >= 0)
                            y[r] = (int)(segrow + (int64_t)pg * a.gs0 +
                                         (int64_t)page_row(p, (int32_t)pos) * a.gs2);
                    }
                }
            };
            int rk_pg = -1, rk_rw = 0, rv_pg0 = -1, rv_rw0 = 0, rv_pg1 = -1, rv_rw1 = 0;
            auto tiled_tile = [&](int64_t tile) { return PG && a.prow > 0 && (tile + 1) * TT <= L; };
            auto page_runs = [&](int64_t tile) {
                rk_pg = -1;
                rk_rw = 0;
                if (lane < TT / a.prow) {
                    const int32_t pos = (int32_t)(tile * TT) + lane * a.prow;
                    const int32_t e = __ldg(p.block_table + (int64_t)b * p.max_pages + page_slot(p, pos));
                    rk_pg = (uint32_t)e < (uint32_t)p.num_pages ? e : -1;
                    if (rk_pg < 0) atomicOr(p.status, kDevBadIndex);
                    rk_rw = page_row(p, pos);
                }
            };
            auto next_rows = [&](int64_t tile) {
                if (tiled_tile(tile)) page_runs(tile); else list_rows(tile, yk);
            };
            if (GA) list_rows(tt0, yk);
            if (PG) next_rows(tt0);
            // masked prefix: which 32-position chunks of a tile some query row
            // sees (bit c = positions 32c .. 32c+31 of the tile as loaded):
            // lane l reads the mask at positions 4l .. 4l+3 for every query
            // index; a position counts if this tile owns it, it lies in the
            // filled prefix (and the causal window) and its mask is not -inf.
            // Hidden chunks are not copied (see the copy step below).
            // The mask values of a tile are loaded one tile before they are
            // evaluated, so the loads never stall the copies.
            const float *mrow = MP ? p.mask + (int64_t)b * p.ms[0] : nullptr;
            constexpr int kMaxQP = 6;
            float mreg[MP ? 4 : 1][MP ? kMaxQP : 1];
            auto mask_load = [&](int64_t tile) {
                const int64_t y0 = tile * TT, ys0 = tile_start(tile, L);
#pragma unroll
                for (int r = 0; r < (MP ? 4 : 1); ++r) {
                    const int64_t pos = ys0 + 4 * lane + r;
                    const bool own = pos >= y0 && pos < L;
#pragma unroll
                    for (int i = 0; i < (MP ? kMaxQP : 1); ++i)
                        mreg[r][i] = own && i < p.n_q ? __ldg(mrow + (int64_t)i * p.ms[1] + pos) : neg_inf();
                }
            };
            auto mask_eval = [&](int64_t tile) -> uint32_t {
                const int64_t ys0 = tile_start(tile, L);
                bool v = false;
#pragma unroll
                for (int r = 0; r < (MP ? 4 : 1); ++r) {
                    const int64_t pos = ys0 + 4 * lane + r;
#pragma unroll
                    for (int i = 0; i < (MP ? kMaxQP : 1); ++i)
                        v = v || (mreg[r][i] != neg_inf() && (!p.causal || pos <= L - p.n_q + i));
                }
                const uint32_t bal = __ballot_sync(0xffffffffu, v);
                uint32_t bits = 0;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) bits |= ((bal >> (8 * cc)) & 0xffu) ? 1u << cc : 0u;
                return bits;
            };
            uint32_t mk_n = 0, mk_v0 = 0, mk_v1 = 0;
            if (MP) {
                mask_load(tt0);
                mk_n = mask_eval(tt0);
                if (n_in > 1) mask_load(tt0 + 1);
            }
            // masked prefix with a chunk list: tile t of the segment is list
            // entries 4t .. 4t+3, chunk c being positions 32c .. 32c+31 of the
            // sequence, loaded as rows min(32c, L - 32) .. + 31 (the last chunk
            // of a length that is no multiple of 32 is right-aligned to end at
            // the length, so nothing past the filled prefix is read).  Lane l
            // holds entry 4 * tile + l for a window of eight tiles (ml_cur) and
            // the next eight (ml_nxt); a copying lane (box cb, chunk cc at lane
            // 4 * cb + cc) keeps its chunk of K(j) for V(j).  An entry outside
            // the prefix's chunks is skipped.
            const int64_t Lr = ML ? seq_len(p, b) : L;     // length of the filled prefix
            const int32_t *mlrow = ML ? p.mlist + (int64_t)b * p.mls : nullptr;
            const int64_t ml_n = L / 32;                    // listed chunks
            const int64_t ml_nch = (Lr + 31) / 32;          // chunks of the prefix
            auto ml_load = [&](int64_t tile) -> int {
                const int64_t e = 4 * tile + lane;
                const int c = e < ml_n ? __ldg(mlrow + e) : -1;
                return c >= 0 && c < ml_nch ? c : -1;
            };
            int ml_cur = -1, ml_nxt = -1, ml_v0 = -1, ml_v1 = -1;
            if (ML) {
                ml_cur = ml_load(tt0);
                if (n_in > 8) ml_nxt = ml_load(tt0 + 8);
            }
            for (int64_t step = 0; step < 2 * n_in && ok; ++step) {
                int64_t j;
                int kv;
                if (step == 0) { j = 0; kv = 0; }
                else if (step == 2 * n_in - 1) { j = n_in - 1; kv = 1; }
                else { j = (step + 1) / 2 - (step & 1 ? 0 : 1); kv = step & 1 ? 0 : 1; }
                const int ys = (int)tile_start(tt0 + j, L);
                if (GA || PG) {
                    // rows of this fill: K(j) takes the prefetched rows (kept
                    // for V(j)), then the next tile's are requested
                    int y[4], rpg = -1, rrw = 0;
                    const bool tl = tiled_tile(tt0 + j);
                    if (kv == 0) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            y[r] = yk[r];
                            if (j & 1) yv1[r] = yk[r]; else yv0[r] = yk[r];
                        }
                        rpg = rk_pg;
                        rrw = rk_rw;
                        if (j & 1) { rv_pg1 = rk_pg; rv_rw1 = rk_rw; } else { rv_pg0 = rk_pg; rv_rw0 = rk_rw; }
                        if (j + 1 < n_in) {
                            if (GA) list_rows(tt0 + j + 1, yk);
                            else next_rows(tt0 + j + 1);
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 4; ++r) y[r] = (j & 1) ? yv1[r] : yv0[r];
                        rpg = (j & 1) ? rv_pg1 : rv_pg0;
                        rrw = (j & 1) ? rv_rw1 : rv_rw0;
                    }
                    const void *map = tl ? (kv ? (const void *)&a.tv : (const void *)&a.tk)
                                         : PG ? (kv ? (const void *)&a.gv : (const void *)&a.gk)
                                              : (kv ? (const void *)&a.tv : (const void *)&a.tk);
                    if (!I8) {
                        const uint32_t slot = issued % C::NS, ph = (issued / C::NS) & 1;
                        if (lane == 0) {
                            ok = bar_wait<I8>(&bs->slot_empty[slot], ph ^ 1, abort_flag, p.wait_ns);
                            if (!ok) note_timeout(bs, p, 1, issued, 0);
                            else ptx::mbar_arrive_expect_tx(&bs->slot_full[slot], C::SLOT);
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (ok && tl) {
                            if (lane < TT / a.prow) {
                                unsigned char *dst = smem + C::OFF_SLOTS + slot * C::SLOT + lane * a.prow * 128;
#pragma unroll
                                for (int cb = 0; cb < C::KB; ++cb)
                                    ptx::tma_load_4d(dst + cb * C::BOX, map, &bs->slot_full[slot], cb * 64,
                                                     rrw, hk, rpg);
                            }
                        } else if (ok) {
                            unsigned char *dst = smem + C::OFF_SLOTS + slot * C::SLOT + 4 * lane * 128;
#pragma unroll
                            for (int cb = 0; cb < C::KB; ++cb)
                                ptx::tma_gather4(dst + cb * C::BOX, map, &bs->slot_full[slot], cb * 64,
                                                 y[0], y[1], y[2], y[3]);
                        }
                    } else {
                        // int8 pages: the four rows' codes (one 128-byte box
                        // each) into the raw ring
                        const uint32_t rs = issued % C::NRX, ph = (issued / C::NRX) & 1;
                        if (lane == 0) {
                            ok = bar_wait<I8>(&bs->raw_empty[rs], ph ^ 1, abort_flag, p.wait_ns);
                            if (!ok) note_timeout(bs, p, 1, issued, 0);
                            else ptx::mbar_arrive_expect_tx(&bs->raw_full[rs], C::RAW);
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        // (one 128-code box per 128 codes of the row: x = 64
                        // pairs apart, TT * 128 bytes apart in the raw tile)
                        if (ok && tl) {
                            if (lane < TT / a.prow) {
#pragma unroll
                                for (int cb = 0; cb < D / 128; ++cb)
                                    ptx::tma_load_4d(smem + C::OFF_RAW + rs * C::RAW + cb * (TT * 128) +
                                                         lane * a.prow * 128,
                                                     map, &bs->raw_full[rs], cb * 64, rrw, hk, rpg);
                            }
                        } else if (ok) {
#pragma unroll
                            for (int cb = 0; cb < D / 128; ++cb)
                                ptx::tma_gather4(smem + C::OFF_RAW + rs * C::RAW + cb * (TT * 128) + 4 * lane * 128,
                                                 map, &bs->raw_full[rs], cb * 64, y[0], y[1], y[2], y[3]);
                        }
                    }
                } else if (MK) {
                    // K(j) takes the chunks found one tile ahead (kept for
                    // V(j)); then the next tile's are read.  (chunk list: the
                    // listed chunks of tile j, the window moving on every
                    // eighth K fill)
                    uint32_t bits;
                    int mc = -1;
                    if (ML) {
                        if (kv == 0) {
                            if (j > 0 && (j & 7) == 0) {
                                ml_cur = ml_nxt;
                                if (j + 8 < n_in) ml_nxt = ml_load(tt0 + j + 8);
                            }
                            mc = __shfl_sync(0xffffffffu, ml_cur, 4 * (int)(j & 7) + (lane & 3));
                            if (j & 1) ml_v1 = mc; else ml_v0 = mc;
                        } else {
                            mc = (j & 1) ? ml_v1 : ml_v0;
                        }
                        bits = __ballot_sync(0xffffffffu, mc >= 0) & 0xfu;
                    } else if (kv == 0) {
                        bits = mk_n;
                        if (j & 1) mk_v1 = bits; else mk_v0 = bits;
                        if (j + 1 < n_in) mk_n = mask_eval(tt0 + j + 1);
                        if (j + 2 < n_in) mask_load(tt0 + j + 2);
                    } else {
                        bits = (j & 1) ? mk_v1 : mk_v0;
                    }
                    const uint32_t slot = issued % C::NS, ph = (issued / C::NS) & 1;
                    // Only the chunks some row sees are loaded; a hidden chunk
                    // keeps the slot's older, finite contents (zeros, or rows
                    // of the filled prefix from an earlier tile), whose scores
                    // are all masked, so their P is zero and the PV adds
                    // nothing.  A tile with no visible chunk loads nothing.
                    if (lane == 0) {
                        ok = bar_wait<I8>(&bs->slot_empty[slot], ph ^ 1, abort_flag, p.wait_ns);
                        if (!ok) note_timeout(bs, p, 1, issued, 0);
                        else if (bits)
                            ptx::mbar_arrive_expect_tx(&bs->slot_full[slot],
                                                       (uint32_t)__popc(bits) * (C::KB * 32 * 128));
                        else
                            ptx::mbar_arrive(&bs->slot_full[slot]);
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    // Four chunks that are consecutive rows (every chunk of a
                    // tile found in place, or four consecutive listed chunks
                    // none of which is a right-aligned last one) are one
                    // 128-row box per 64 columns (maps gk / gv); otherwise
                    // lane 4*cb + cc copies 32 rows (chunk cc) of box cb.
                    bool whole = bits == 0xfu;
                    int row0 = ys;
                    if (ML) {
                        row0 = 32 * __shfl_sync(0xffffffffu, mc, 0);
                        whole = __all_sync(0xffffffffu, mc == row0 / 32 + (lane & 3)) && row0 >= 0 &&
                                (int64_t)row0 + TT <= Lr;
                    }
                    if (ok && whole) {
                        if (lane < C::KB)
                            ptx::tma_load_4d(smem + C::OFF_SLOTS + slot * C::SLOT + lane * C::BOX,
                                             kv ? (const void *)&a.gv : (const void *)&a.gk,
                                             &bs->slot_full[slot], lane * 64, row0, hk, b);
                    } else if (ok && lane < 4 * C::KB && ((bits >> (lane & 3)) & 1u)) {
                        const int cb = lane >> 2, cc = lane & 3;
                        const int row = ML ? (int)min((int64_t)32 * mc, Lr - 32) : ys + 32 * cc;
                        ptx::tma_load_4d(smem + C::OFF_SLOTS + slot * C::SLOT + cb * C::BOX + cc * (32 * 128),
                                         kv ? (const void *)&a.tv : (const void *)&a.tk,
                                         &bs->slot_full[slot], cb * 64, row, hk, b);
                    }
                } else if (lane == 0 && I8) {
                    // int8 codes -> raw ring (one box of TT positions x D codes)
                    const uint32_t rs = issued % C::NRX, ph = (issued / C::NRX) & 1;
                    ok = bar_wait<I8>(&bs->raw_empty[rs], ph ^ 1, abort_flag, p.wait_ns);
                    if (!ok) note_timeout(bs, p, 1, issued, 0);
                    if (ok) {
                        ptx::mbar_arrive_expect_tx(&bs->raw_full[rs], C::RAW);
#pragma unroll
                        for (int cb = 0; cb < D / 128; ++cb)
                            ptx::tma_load_4d(smem + C::OFF_RAW + rs * C::RAW + cb * (TT * 128),
                                             kv ? (const void *)&a.tv : (const void *)&a.tk,
                                             &bs->raw_full[rs], cb * 64, ys, hkc, b);
                    }
                } else if (lane == 0) {
                    const uint32_t slot = issued % C::NS, ph = (issued / C::NS) & 1;
                    ok = bar_wait<I8>(&bs->slot_empty[slot], ph ^ 1, abort_flag, p.wait_ns);
                    if (!ok) note_timeout(bs, p, 1, issued, 0);
                    if (ok) {
                        ptx::mbar_arrive_expect_tx(&bs->slot_full[slot], C::SLOT);
                        unsigned char *dst = smem + C::OFF_SLOTS + slot * C::SLOT;
#pragma unroll
                        for (int cb = 0; cb < C::KB; ++cb)
                            ptx::tma_load_4d(dst + cb * C::BOX, kv ? (const void *)&a.tv
                                                                   : (const void *)&a.tk,
                                             &bs->slot_full[slot], cb * 64, ys, hk, b);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok) ++issued;
            }
            ++piece;
            if (piece_end >= t_end || !next_piece(p, w) || w.first >= t_end) break;
            t = w.first;
        }
        // Drain: every issued copy must land before the block exits.
        if (lane == 0) {
            constexpr uint32_t RING = I8 ? (uint32_t)C::NRX : (uint32_t)C::NS;
            const uint32_t n = issued < RING ? issued : RING;
            for (uint32_t k = 0; k < n; ++k) {
                const uint32_t idx = issued - 1 - k;
                ptx::mbar_wait_drain(I8 ? &bs->raw_full[idx % RING] : &bs->slot_full[idx % RING],
                                     (idx / RING) & 1, kWaitNs);
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA issuer
        uint32_t tile_ctr = 0;
        int piece = 0;
        bool ok = true;
        bool issued_any = false;
        uint32_t pa = 0, pb = 0;   // first and last tile number of the current piece
        // S^T[pos, row] = sum_d K[pos, d] Q[row, d] for tile number tc.
        auto issue_qk = [&](uint32_t tc) -> bool {
            const uint32_t sb = tc & 1, u = tc >> 1, ki = k_fill(tc, pa), ks = ki % C::NS;
            if (!bar_wait<I8>(&bs->slot_full[ks], (ki / C::NS) & 1, abort_flag, p.wait_ns)) {
                note_timeout(bs, p, 3, tc, piece);
                return false;
            }
            if (!bar_wait<I8>(&bs->s_free[sb], (u & 1) ^ 1, abort_flag, p.wait_ns)) {
                note_timeout(bs, p, 4, tc, piece);
                return false;
            }
            ptx::tc_fence_after();
            const uint32_t k_addr = smem_base + C::OFF_SLOTS + ks * C::SLOT;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t da = ptx::smem_desc(k_addr + (kk >> 2) * C::BOX + (kk & 3) * 32, 16,
                                                   1024, ptx::kLayoutSwizzle128);
                const uint64_t db = ptx::smem_desc(q_addr + (kk >> 2) * C::QB + (kk & 3) * 32, 16,
                                                   1024, ptx::kLayoutSwizzle128);
                ptx::mma_f16_ss(tmem + sb * N, da, db, C::IDESC_QK, kk > 0);
            }
            ptx::mma_commit(&bs->slot_empty[ks]);
            ptx::mma_commit(&bs->s_full[sb]);
            issued_any = true;
            return true;
        };
        // O^T[dim, row] += sum_pos V[pos, dim] (P_hi + P_lo)[row, pos] for tile tc.
        auto issue_pv = [&](uint32_t tc, bool first) -> bool {
            const uint32_t vi = v_fill(tc, pb), vs = vi % C::NS;
            const uint32_t ps = tc % C::PST, pu = tc / C::PST;
            if (!bar_wait<I8>(&bs->slot_full[vs], (vi / C::NS) & 1, abort_flag, p.wait_ns)) {
                note_timeout(bs, p, 6, tc, piece);
                return false;
            }
            if (!bar_wait<I8>(&bs->p_full[ps], pu & 1, abort_flag, p.wait_ns)) {
                note_timeout(bs, p, 7, tc, piece);
                return false;
            }
            ptx::tc_fence_after();
            const uint32_t v_addr = smem_base + C::OFF_SLOTS + vs * C::SLOT;
            const uint32_t pb = p_addr + ps * C::PSTAGE;
            const bool two_planes = p.out_f32 != 0;
            // O^T += V^T P_hi^T (+ V^T P_lo^T for fp32 outputs)
            auto pv_tiles = [&](auto planes) {
                constexpr int NP = decltype(planes)::value;
#pragma unroll
                for (int dc = 0; dc < C::DC; ++dc) {
#pragma unroll
                    for (int kt = 0; kt < TT / 16; ++kt) {
                        const uint64_t da = ptx::smem_desc(v_addr + (2 * dc) * C::BOX + kt * 2048,
                                                           C::BOX, 1024, ptx::kLayoutSwizzle128);
#pragma unroll
                        for (int pl = 0; pl < NP; ++pl) {
                            const uint64_t db = ptx::smem_desc(pb + pl * C::PPLANE + kt * 512,
                                                               C::PATOM, 256, ptx::kLayoutSwizzle32);
                            ptx::mma_f16_ss(tmem + 2 * N + dc * N, da, db, C::IDESC_PV,
                                            (first && kt == 0 && pl == 0) ? 0u : 1u);
                        }
                    }
                }
            };
            if (two_planes) pv_tiles(std::integral_constant<int, 2>());
            else pv_tiles(std::integral_constant<int, 1>());
            ptx::mma_commit(&bs->slot_empty[vs]);
            ptx::mma_commit(&bs->p_free[ps]);
            ptx::mma_commit(&bs->o_done);
            return true;
        };
        Walk w = bs->walk;
        int64_t t = max(t_begin, w.first);
        while (ok) {
            const int64_t piece_end = min(t_end, w.first + w.ntiles);
            const uint32_t n_in = (uint32_t)(piece_end - t);
            pa = tile_ctr;
            pb = tile_ctr + n_in - 1;
            if (lane == 0) {
                // Software pipeline: QK of tile j+1 is issued before PV of
                // tile j, so the next scores are ready when softmax finishes.
                // (int8 caches: once the widening threads have converted Q)
                ok = bar_wait<I8>(I8 ? &bs->q_conv : &bs->q_full, piece & 1, abort_flag, p.wait_ns);
                if (!ok) note_timeout(bs, p, 2, tile_ctr, piece);
                ptx::tc_fence_after();
                ok = ok && issue_qk(tile_ctr);
                if (ok && n_in == 1) ptx::mma_commit(&bs->q_free);
                for (uint32_t j = 0; j < n_in && ok; ++j) {
                    if (j + 1 < n_in) {
                        ok = issue_qk(tile_ctr + j + 1);
                        if (!ok) break;
                        if (j + 2 == n_in) ptx::mma_commit(&bs->q_free);
                    }
                    if (j == 0 && piece > 0) {
                        ok = bar_wait<I8>(&bs->o_free, (piece - 1) & 1, abort_flag, p.wait_ns);
                        if (!ok) note_timeout(bs, p, 5, tile_ctr, piece);
                    }
                    ok = ok && issue_pv(tile_ctr + j, j == 0);
                }
                if (!ok) set_abort(bs, p);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            tile_ctr += n_in;
            ++piece;
            if (piece_end >= t_end || !next_piece(p, w) || w.first >= t_end) break;
            t = w.first;
        }
        // Drain: all MMAs issued by this thread complete before TMEM is freed.
        if (lane == 0 && issued_any) {
            ptx::mma_commit(&bs->exit_mma);
            ptx::mbar_wait_drain(&bs->exit_mma, 0, kWaitNs);
        }
    } else if (I8 && warp >= 4) {
        // ------------------------------------- int8 -> fp16 widening (warps 4-7)
        // Fill f of the raw ring becomes fill f of the fp16 slot ring, in the
        // producer's order.  Codes widen exactly (fp16 holds every integer
        // of magnitude <= 2048), two instructions per pair of codes; the
        // per-position scales are applied to the scores and to P by the
        // softmax group, so nothing here rounds.  Raw tile: row-major
        // [TT][D] codes.  fp16 tile: KB boxes of [TT][64] with the 128-byte
        // swizzle (16-byte chunk c of position r at c ^ (r & 7)), the layout
        // of a TMA load of a 16-bit cache.
        const int ct = tid - 128;
        uint32_t f = 0;
        bool ok = true;
        int piece = 0;
        Walk w = bs->walk;
        int64_t t = max(t_begin, w.first);
        while (ok) {
            const int64_t piece_end = min(t_end, w.first + w.ntiles);
            const int64_t n_fill = 2 * (piece_end - t);
            // The piece's Q (bf16, as the producer loaded it) -> fp16 in place
            // (exact for normal values up to 65504, saturating beyond); the
            // MMA issuer waits for q_conv.  Padding rows are zeros either way.
            ok = bar_wait<I8>(&bs->q_full, piece & 1, abort_flag, p.wait_ns);
            if (!ok) { note_timeout(bs, p, 19, f, piece); break; }
            for (uint32_t e = ct; e < C::QBYTES / 16; e += 128) {
                uint4 *q4 = reinterpret_cast<uint4 *>(smem + C::OFF_Q) + e;
                const uint4 v = *q4;
                *q4 = make_uint4(pack_f16x2(bf16lo(v.x), bf16hi(v.x)), pack_f16x2(bf16lo(v.y), bf16hi(v.y)),
                                 pack_f16x2(bf16lo(v.z), bf16hi(v.z)), pack_f16x2(bf16lo(v.w), bf16hi(v.w)));
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bs->q_conv);
            for (int64_t k = 0; k < n_fill && ok; ++k, ++f) {
                const uint32_t rs = f % C::NRX, ss = f % C::NS;
                ok = bar_wait<I8>(&bs->raw_full[rs], (f / C::NRX) & 1, abort_flag, p.wait_ns);
                if (!ok) { note_timeout(bs, p, 17, f, piece); break; }
                // Thread ct takes 16 codes (dims 16*q16 .. 16*q16+15) of
                // positions r0 + RSTEP*k: one 16-byte load and two swizzled
                // 16-byte stores each, all loads issued first.  Each group of
                // 8 threads covers half of two rows (of one 128-code box of
                // them), its low half of one and high half of the other, so
                // its 8 loads and each of its two sets of 8 stores fall in 8
                // different bank groups.
                // Raw tile: RB boxes of [TT][128] codes, 128-byte swizzled
                // (chunk c of row r at c ^ (r & 7)); head_dim 256 rows span
                // two boxes, taken by alternate pairs of 8-thread groups.
                constexpr int RB = D / 128, RSTEP = 16 / RB, NK = TT / RSTEP;
                static_assert(!I8 || D == 128 || D == 256, "int8 tiles: head_dim 128 or 256");
                const int quarter = ct >> 3, tq = ct & 7;
                const int rbox = RB == 1 ? 0 : (quarter >> 1) & 1;
                const int r0 = 2 * (quarter >> (RB == 1 ? 1 : 2)) + (tq >> 2);
                const int c8 = (tq & 3) + 4 * ((tq >> 2) ^ (quarter & 1));
                const int q16 = rbox * 8 + c8;    // 16-code group of the row
                const unsigned char *raw = smem + C::OFF_RAW + rs * C::RAW + rbox * (TT * 128) +
                                           r0 * 128 + ((c8 ^ (r0 & 7)) << 4);
                unsigned char *dst = smem + C::OFF_SLOTS + ss * C::SLOT + (q16 >> 2) * C::BOX +
                                     r0 * 128;
                // (r0 + RSTEP*k) & 7 == r0 & 7: the swizzled chunk offsets are per thread
                const int sw0 = (((2 * q16) & 7) ^ (r0 & 7)) << 4, sw1 = (((2 * q16 + 1) & 7) ^ (r0 & 7)) << 4;
                uint4 cw[NK];
#pragma unroll
                for (int k = 0; k < NK; ++k)
                    cw[k] = *reinterpret_cast<const uint4 *>(raw + k * RSTEP * 128);
                // The raw slot is free for the next copy once the codes are
                // in registers; then wait for an fp16 slot the MMAs released.
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&bs->raw_empty[rs]);
                ok = bar_wait<I8>(&bs->slot_empty[ss], ((f / C::NS) & 1) ^ 1, abort_flag, p.wait_ns);
                if (!ok) { note_timeout(bs, p, 18, f, piece); break; }
#pragma unroll
                for (int k = 0; k < NK; ++k) {
                    unsigned char *row = dst + k * RSTEP * 128;
                    const uint32_t ux = cw[k].x ^ 0x80808080u, uy = cw[k].y ^ 0x80808080u;
                    const uint32_t uz = cw[k].z ^ 0x80808080u, uw = cw[k].w ^ 0x80808080u;
                    *reinterpret_cast<uint4 *>(row + sw0) =
                        make_uint4(i8x2_to_f16x2(ux, 0), i8x2_to_f16x2(ux, 2),
                                   i8x2_to_f16x2(uy, 0), i8x2_to_f16x2(uy, 2));
                    *reinterpret_cast<uint4 *>(row + sw1) =
                        make_uint4(i8x2_to_f16x2(uz, 0), i8x2_to_f16x2(uz, 2),
                                   i8x2_to_f16x2(uw, 0), i8x2_to_f16x2(uw, 2));
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&bs->slot_full[ss]);
            }
            if (!ok) { set_abort(bs, p); break; }
            ++piece;
            if (piece_end >= t_end || !next_piece(p, w) || w.first >= t_end) break;
            t = w.first;
        }
    } else {
        // ------------------------------------------- softmax and epilogue
        // Two warpgroups split the query rows: group wg owns rows
        // [wg*NH, wg*NH + NH), i.e. those columns of S^T, O^T and P.  Thread
        // wt of a group owns TMEM lane wt: cache position wt of the tile.
        constexpr int NH = C::NH;
        const int wg = warp >> 2, wwarp = warp & 3, wt = tid & 127;
        const int cb0 = wg * NH;                  // first row (column) of the group
        const uint32_t lane_base = (uint32_t)(wwarp * 32) << 16;
        float *gred = red + wg * C::RED_GROUP;    // the group's reduction scratch
        uint32_t tile_ctr = 0;
        uint32_t o_seen = 0;      // o_done phases observed, consumed strictly in order
        uint32_t wg_ctr = 0;      // uses of the group barrier
        uint32_t sm_ctr = 0;      // uses of the two-group barrier
        int piece = 0;
        bool ok = true;
        // Completion of PV number k (k = 0, 1, ...), phase by phase.  Every
        // tile consumes the previous tile's phase before publishing its own P,
        // so the barrier is never more than one phase ahead of this wait and
        // the parity test cannot alias.
        auto wait_pv = [&](uint32_t k) -> bool {
            for (; o_seen <= k; ++o_seen)
                if (!bar_wait<(I8 && NV <= 8)>(&bs->o_done, o_seen & 1, abort_flag, p.wait_ns)) {
                    note_timeout(bs, p, 11, tile_ctr, piece);
                    return false;
                }
            return true;
        };
        // Barrier over this warpgroup's 128 threads, bounded.
        auto wg_sync = [&]() -> bool {
            ptx::mbar_arrive(&bs->wg_bar[wg]);
            if (bar_wait<(I8 && NV <= 8)>(&bs->wg_bar[wg], (wg_ctr++) & 1, abort_flag, p.wait_ns)) return true;
            note_timeout(bs, p, 10, tile_ctr, piece);
            return false;
        };
        // Barrier over both warpgroups, bounded.
        auto sm_sync = [&]() -> bool {
            ptx::mbar_arrive(&bs->sm_bar);
            if (bar_wait<(I8 && NV <= 8)>(&bs->sm_bar, (sm_ctr++) & 1, abort_flag, p.wait_ns)) return true;
            note_timeout(bs, p, 14, tile_ctr, piece);
            return false;
        };
        Walk w = bs->walk;
        int64_t t = max(t_begin, w.first);
        while (ok) {
            const int64_t s = w.s;
            const int64_t piece_end = min(t_end, w.first + w.ntiles);
            const int64_t n_in = piece_end - t;
            const int64_t tt0 = t - w.first;
            const int64_t L = w.L;
            const int64_t Lr = ML ? seq_len(p, w.b) : L;    // length of the filled prefix
            const int rows = p.rows;

            // Output offsets of this group's rows (one division sequence per
            // row, so the unrolled per-row code below needs none) and the
            // causal limit of each row.  The Q rows arrive by TMA.
            int64_t *ooff = otbl + (piece & 1) * N;
            if (share_merge && tid == 0) bs->walk_last = w;
            if (wt < NH && cb0 + wt < rows) {
                // (gather: the list's query row, head offset r)
                const int r = cb0 + wt;
                const int i = GA ? w.i : r % p.n_q, h = w.hk * p.g + (GA ? r : r / p.n_q);
                ooff[r] = (int64_t)w.b * p.os[0] + (int64_t)i * p.os[1] + (int64_t)h * p.os[2];
            }
            int lim[NH];    // last visible position of each row
            {
                int qi = cb0 % p.n_q;
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    lim[r] = p.causal ? (int)(Lr - p.n_q + qi) : (int)(Lr - 1);
                    if (++qi == p.n_q) qi = 0;
                }
            }

            float mrun[NH], lpart[NH];
#pragma unroll
            for (int r = 0; r < NH; ++r) { mrun[r] = neg_inf(); lpart[r] = 0.f; }

            // int8 caches: this segment's per-position scales, read one tile
            // ahead (k scale multiplies the scores, v scale multiplies P but
            // not the row sums; nothing outside the filled prefix is read).
            // (paged: scales live beside their rows, page pg_n, row tok % page_size)
            const int64_t sb0 = PG ? 0 : (int64_t)w.b;
            const int64_t hkc = (I8 && !GA && !PG) && p.kvdiv > 1 ? w.hk / p.kvdiv : w.hk;
            const float *ksrow = I8 ? p.k_scale + sb0 * p.kss[0] + hkc * p.kss[1] : nullptr;
            const float *vsrow = I8 ? p.v_scale + sb0 * p.vss[0] + hkc * p.vss[1] : nullptr;
            // paged: the pool page of this thread's position (-1 past the
            // length, or for a table entry outside the pool, which the
            // producer flags), read two tiles ahead so the scale reads of the
            // next tile need not wait for it: pg_c for tile j, pg_n for j + 1
            const int32_t *trow = PG ? p.block_table + (int64_t)w.b * p.max_pages : nullptr;
            auto page_at = [&](int64_t jj) -> int {
                const int32_t tok = (int32_t)((tt0 + jj) * TT) + wt;
                if (tok >= (int32_t)L) return -1;
                const int32_t e = __ldg(trow + page_slot(p, tok));
                return (uint32_t)e < (uint32_t)p.num_pages ? e : -1;
            };
            int pg_c = -1, pg_n = -1;
            if (PG) {
                pg_c = page_at(0);
                if (n_in > 1) pg_n = page_at(1);
            }
            float ksc_n = 1.f, vsc_n = 1.f;
            // (gather over int8 caches: the scales of the list's cells, the
            // cell of a tile being read one tile before its scales)
            int cell_nn = -1;
            auto load_scales = [&](int64_t jj, int pg) {
                if (GA) {
                    if (pg >= 0 && pg < p.cap) {
                        ksc_n = __ldg(ksrow + (int64_t)pg * p.kss[2]);
                        vsc_n = __ldg(vsrow + (int64_t)pg * p.vss[2]);
                    }
                } else if (PG) {
                    const int64_t tok = (tt0 + jj) * TT + wt;
                    if (pg >= 0) {
                        const int64_t r = page_row(p, (int32_t)tok);
                        ksc_n = __ldg(ksrow + (int64_t)pg * p.kss[0] + r * p.kss[2]);
                        vsc_n = __ldg(vsrow + (int64_t)pg * p.vss[0] + r * p.vss[2]);
                    }
                } else {
                    const int64_t tok = tile_start(tt0 + jj, L) + wt;
                    if (tok >= (tt0 + jj) * TT && tok < L) {
                        ksc_n = __ldg(ksrow + tok * p.kss[2]);
                        vsc_n = __ldg(vsrow + tok * p.vss[2]);
                    }
                }
            };
            if (I8 && !GA) load_scales(0, pg_c);
            // gather: the list cell this lane's position holds, read one tile
            // ahead; a cell is visible if 0 <= cell < cap (cap or more is
            // flagged FD_DEV_BAD_INDEX, negative is padding).
            // With a bias list, the entry's bias (log2 units) rides along;
            // -inf drops the entry.
            const int32_t *ilist = GA ? p.idx + ((int64_t)w.b * p.n_q + w.i) * p.idx_len : nullptr;
            const float *blist =
                GA && p.bias ? p.bias + ((int64_t)w.b * p.n_q + w.i) * p.idx_len : nullptr;
            int cell_n = -1;
            float bias_n = 0.f;
            auto list_cell = [&](int64_t jj) -> int {
                const int64_t pos = (tt0 + jj) * TT + wt;
                return pos < p.idx_len ? __ldg(ilist + pos) : -1;
            };
            auto load_cell = [&](int64_t jj) {
                const int64_t pos = (tt0 + jj) * TT + wt;
                cell_n = list_cell(jj);
                if (blist) bias_n = pos < p.idx_len ? __ldg(blist + pos) : 0.f;
            };
            if (GA) load_cell(0);
            if (GA && I8) {
                if (n_in > 1) cell_nn = list_cell(1);
                load_scales(0, cell_n);
            }
            // masked prefix: this position's mask value (log2 units, -inf
            // hides it) for each query index, read one tile ahead
            constexpr int kMaxQ = 6;
            const float *mrow = MK ? p.mask + (int64_t)w.b * p.ms[0] : nullptr;
            float mk_n[kMaxQ];
            // chunk list: warp wwarp holds positions 32 * wwarp .. + 31 of a
            // tile, the chunk of list entry 4 * tile + wwarp, loaded as rows
            // min(32c, Lr - 32) .. + 31, of which it owns those at or past 32c;
            // the chunk of tile j + 1 is read during tile j - 1, its mask
            // values during tile j
            const int32_t *mlrow = ML ? p.mlist + (int64_t)w.b * p.mls : nullptr;
            const int64_t ml_n = L / 32, ml_nch = (Lr + 31) / 32;
            auto ml_chunk = [&](int64_t jj) -> int {
                const int64_t e = 4 * (tt0 + jj) + wwarp;
                const int c = e < ml_n ? __ldg(mlrow + e) : -1;
                return c >= 0 && c < ml_nch ? c : -1;
            };
            auto ml_token = [&](int c) -> int64_t {
                return c >= 0 ? min((int64_t)32 * c, Lr - 32) + lane : -1;
            };
            int mc_j = -1, mc_j1 = -1;    // chunks of tiles j and j + 1
            if (ML) {
                mc_j = ml_chunk(0);
                if (n_in > 1) mc_j1 = ml_chunk(1);
            }
            auto load_mask = [&](int64_t jj, int c) {
                int64_t tok;
                bool own;
                if (ML) {
                    tok = ml_token(c);
                    own = c >= 0 && tok >= (int64_t)32 * c;
                } else {
                    tok = tile_start(tt0 + jj, L) + wt;
                    own = tok >= (tt0 + jj) * TT && tok < L;
                }
#pragma unroll
                for (int i = 0; i < kMaxQ; ++i)
                    mk_n[i] = own && i < p.n_q ? __ldg(mrow + (int64_t)i * p.ms[1] + tok) * 1.4426950408889634f
                                               : neg_inf();
            };
            if (MK) load_mask(0, mc_j);
            for (int64_t j = 0; j < n_in && ok; ++j) {
                const int64_t y0 = (tt0 + j) * TT;
                const int64_t token = ML ? ml_token(mc_j) : (GA || PG) ? y0 + wt : tile_start(tt0 + j, L) + wt;
                const uint32_t sb = tile_ctr & 1, u = tile_ctr >> 1;
                // Visibility: a position this tile owns (the right-aligned last
                // tile also holds positions the previous tile covered), inside
                // the filled prefix and, for causal windows, at or before
                // L - n_q + i for the row's query index i.  Gather: a valid
                // cell of the list.  Paged: a position on a page of the pool.
                bool in_len = ML ? mc_j >= 0 && token >= (int64_t)32 * mc_j : token >= y0 && token < L;
                float bl = 0.f;
                if (GA) {
                    const int cell = cell_n;
                    const float cb = bias_n;
                    if (I8) {
                        cell_n = cell_nn;
                        if (j + 2 < n_in) cell_nn = list_cell(j + 2);
                    } else if (j + 1 < n_in) {
                        load_cell(j + 1);
                    }
                    if (cell >= p.cap) atomicOr(p.status, kDevBadIndex);
                    in_len = in_len && cell >= 0 && cell < p.cap && cb != neg_inf();
                    bl = cb * 1.4426950408889634f;
                }
                const int pg_next = pg_n;
                if (PG) {
                    in_len = in_len && pg_c >= 0;
                    if (j + 2 < n_in) pg_n = page_at(j + 2);
                }
                float mk[kMaxQ];
                if (MK) {
#pragma unroll
                    for (int i = 0; i < kMaxQ; ++i) mk[i] = mk_n[i];
                    if (j + 1 < n_in) load_mask(j + 1, mc_j1);
                    if (ML) {
                        mc_j = mc_j1;
                        mc_j1 = j + 2 < n_in ? ml_chunk(j + 2) : -1;
                    }
                }
                const float ksc = ksc_n, vsc = vsc_n;
                if (I8 && j + 1 < n_in) load_scales(j + 1, GA ? cell_n : pg_next);
                pg_c = pg_next;
                ok = bar_wait<(I8 && NV <= 8)>(&bs->s_full[sb], u & 1, abort_flag, p.wait_ns);
                if (!ok) { note_timeout(bs, p, 9, tile_ctr, piece); break; }
                ptx::tc_fence_after();
                float sv[NH];
                ptx::tmem_ld_cols<NH>(tmem + lane_base + sb * N + cb0, sv);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bs->s_free[sb]);

                const float sl = I8 ? p.scale_log2 * ksc : p.scale_log2;
                int mq = cb0 % p.n_q;   // masked prefix: query index of row r
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    bool vis = in_len && cb0 + r < rows && token <= lim[r];
                    if (GA) {
                        sv[r] = vis ? __fmaf_rn(sv[r], sl, bl) : neg_inf();
                    } else if (MK) {
                        float mb = mk[0];
#pragma unroll
                        for (int i = 1; i < kMaxQ; ++i) mb = mq == i ? mk[i] : mb;
                        vis = vis && mb != neg_inf();
                        sv[r] = vis ? __fmaf_rn(sv[r], sl, mb) : neg_inf();
                        if (++mq == p.n_q) mq = 0;
                    } else {
                        sv[r] = vis ? sv[r] * sl : neg_inf();
                    }
                }
                // Refresh the running maxima only when some score passes
                // mrun + kRescaleSlack (always on a segment's first tile).
                bool need = false;
#pragma unroll
                for (int r = 0; r < NH; ++r) need = need || (sv[r] > mrun[r] + C::SLACK);
                need = __any_sync(0xffffffffu, need);
                if (lane == 0) bs->vote[wg][tile_ctr & 1][wwarp] = need;
                ok = wg_sync();
                if (!ok) break;
                const int *vt = bs->vote[wg][tile_ctr & 1];
                if (vt[0] | vt[1] | vt[2] | vt[3]) {
                    // Column maxima over the 128 positions of the tile.
                    float *rb = gred + (tile_ctr & 1) * (4 * NH);
#pragma unroll
                    for (int r = 0; r < NH; ++r) {
                        const float mx = warp_max(sv[r]);
                        if (lane == 0) rb[wwarp * NH + r] = mx;
                    }
                    ok = wg_sync();
                    if (!ok) break;
                    float alpha[NH];
                    bool grow = false;
#pragma unroll
                    for (int r = 0; r < NH; ++r) {
                        const float tmax = fmaxf(fmaxf(rb[r], rb[NH + r]),
                                                 fmaxf(rb[2 * NH + r], rb[3 * NH + r]));
                        // Only rows that passed their own threshold move,
                        // so a row's arithmetic never depends on another
                        // row's scores.
                        const float mnew = tmax > mrun[r] + C::SLACK ? tmax : mrun[r];
                        const float muse = mnew == neg_inf() ? 0.f : mnew;
                        alpha[r] = fast_exp2(mrun[r] - muse);
                        grow = grow || (alpha[r] < 1.f);
                        mrun[r] = mnew;
                        lpart[r] *= alpha[r];
                    }
                    // Rescale this group's columns of the running O in TMEM
                    // (after the previous PV landed).
                    if (grow && j > 0) {
                        ok = wait_pv(tile_ctr - 1);
                        if (!ok) break;
                        ptx::tc_fence_after();
#pragma unroll
                        for (int dc = 0; dc < C::DC; ++dc) {
                            float o[NH];
                            const uint32_t ta = tmem + lane_base + 2 * N + dc * N + cb0;
                            ptx::tmem_ld_cols<NH>(ta, o);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < NH; ++k) o[k] *= alpha[k];
                            ptx::tmem_st_cols<NH>(ta, o);
                        }
                        ptx::tmem_wait_st();
                    }
                }
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    const float muse = mrun[r] == neg_inf() ? 0.f : mrun[r];
                    const float pr = fast_exp2(sv[r] - muse);
                    lpart[r] += pr;
                    sv[r] = I8 ? pr * vsc : pr;
                }
                // P^T for the PV product.
                const uint32_t ps = tile_ctr % C::PST, pu = tile_ctr / C::PST;
                ok = bar_wait<(I8 && NV <= 8)>(&bs->p_free[ps], (pu & 1) ^ 1, abort_flag, p.wait_ns);
                if (!ok) { note_timeout(bs, p, 13, tile_ctr, piece); break; }
                // PV of the previous tile must have completed before P of this
                // tile is published (see wait_pv).
                if (tile_ctr > 0) {
                    ok = wait_pv(tile_ctr - 1);
                    if (!ok) break;
                }
                {
                    // P = hi + lo, both bf16: hi = rn(p), lo = rn(p - hi), so the
                    // PV product sees p to about 2^-17 relative, which fp32
                    // outputs need; bf16 outputs (2^-9 themselves) take P_hi
                    // alone, which halves the PV MMAs.  (int8 caches: both
                    // fp16, about 2^-22 relative, p carrying the v scale.)  Thread wt
                    // writes its position's row: 8 query rows per 16-byte chunk,
                    // chunk c of a 16-row atom stored at c ^ bit 2 of wt.
                    unsigned char *prow = smem + C::OFF_P + ps * C::PSTAGE + wt * 32;
                    const int sw = (wt >> 2) & 1;
#pragma unroll
                    for (int l8 = 0; l8 < NH / 8; ++l8) {
                        const int a8 = cb0 / 8 + l8;      // global 8-row group
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float p0 = sv[l8 * 8 + 2 * e], p1 = sv[l8 * 8 + 2 * e + 1];
                            if (I8) {   // fp16 planes (int8 caches)
                                const uint32_t h = pack_f16x2(p0, p1);
                                hw[e] = h;
                                lw[e] = pack_f16x2(p0 - f16lo(h), p1 - f16hi(h));
                            } else {
                                const uint32_t h = pack_bf16x2(p0, p1);
                                hw[e] = h;
                                lw[e] = pack_bf16x2(p0 - bf16lo(h), p1 - bf16hi(h));
                            }
                        }
                        const uint32_t off = (a8 >> 1) * C::PATOM + (((a8 & 1) ^ sw) << 4);
                        *reinterpret_cast<uint4 *>(prow + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        if (p.out_f32)
                            *reinterpret_cast<uint4 *>(prow + C::PPLANE + off) =
                                make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bs->p_full[ps]);
                ++tile_ctr;
            }
            if (!ok) { set_abort(bs, p); break; }

            // ------------------------------------------ segment epilogue
            ok = wait_pv(tile_ctr - 1);
            if (!ok) { set_abort(bs, p); break; }
            ptx::tc_fence_after();
            float o[C::DC][NH];
#pragma unroll
            for (int dc = 0; dc < C::DC; ++dc)
                ptx::tmem_ld_cols<NH>(tmem + lane_base + 2 * N + dc * N + cb0, o[dc]);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bs->o_free);

            // Row sums of P over the segment piece (this group's rows).
            float *lb = gred + (tile_ctr & 1) * (4 * NH);
#pragma unroll
            for (int r = 0; r < NH; ++r) {
                const float v = warp_sum(lpart[r]);
                if (lane == 0) lb[wwarp * NH + r] = v;
            }
            ok = wg_sync();
            float lsum[NH];
#pragma unroll
            for (int r = 0; r < NH; ++r) lsum[r] = lb[r] + lb[NH + r] + lb[2 * NH + r] + lb[3 * NH + r];
            ok = ok && wg_sync();
            if (!ok) { set_abort(bs, p); break; }

            // Blocks sharing the segment (owner() only where the piece is
            // cut at this block's range boundary).
            const int c_first = CL ? c : w.first >= t_begin ? c : sp.owner(w.first);
            const int c_last = CL ? c : w.first + w.ntiles <= t_end ? c : sp.owner(w.first + w.ntiles - 1);
            if (CL) {
                // the partial (O, m, l) stays in this block's K/V slots, idle
                // after its only piece, for the cluster's merge at the end
                float *part = reinterpret_cast<float *>(smem + C::OFF_SLOTS);
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    if (cb0 + r < rows) {
#pragma unroll
                        for (int dc = 0; dc < C::DC; ++dc) part[(cb0 + r) * D + dc * 128 + wt] = o[dc][r];
                    }
                }
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    if (r == wt && cb0 + r < rows) {
                        part[rows * D + cb0 + r] = mrun[r];
                        part[rows * D + rows + cb0 + r] = lsum[r];
                    }
                }
            } else if (c_first == c_last) {
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    if (cb0 + r < rows) {
                        const float inv = lsum[r] > 0.f ? 1.f / lsum[r] : 0.f;
                        const int64_t off = ooff[cb0 + r];
#pragma unroll
                        for (int dc = 0; dc < C::DC; ++dc) {
                            const float val = o[dc][r] * inv;
                            if (p.out_f32)
                                reinterpret_cast<float *>(p.out)[off + dc * 128 + wt] = val;
                            else
                                reinterpret_cast<uint16_t *>(p.out)[off + dc * 128 + wt] = bf16_bits(val);
                        }
                    }
                }
            } else {
                float *slot = slot_ptr(p, s, c);
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    if (cb0 + r < rows) {
#pragma unroll
                        for (int dc = 0; dc < C::DC; ++dc)
                            slot[(cb0 + r) * D + dc * 128 + wt] = o[dc][r];
                    }
                }
                // every thread of the group holds the same mrun / lsum values
#pragma unroll
                for (int r = 0; r < NH; ++r) {
                    if (r == wt && cb0 + r < rows) {
                        slot[rows * D + cb0 + r] = mrun[r];
                        slot[rows * D + rows + cb0 + r] = lsum[r];
                    }
                }
                __threadfence();
                ok = sm_sync();
                if (tid == 0 && ok) bs->last_flag = atomicAdd(p.counters + s, 1) == c_last - c_first;
                ok = ok && sm_sync();
                if (!ok) { set_abort(bs, p); break; }
                const int r1w = min(cb0 + NH, rows);       // this group merges rows cb0 .. r1w-1
                if (!share_merge && bs->last_flag && r1w > cb0) {
                    __threadfence();
                    if constexpr (I8 && NV <= 8 && !GA && !PG)
                        merge_split_rows_ool<D, NH, C::MERGE_UNROLL>(p, s, c_first, c_last, cb0, r1w, wt, ooff);
                    else
                        merge_split_rows<D, NH, C::MERGE_UNROLL>(p, s, c_first, c_last, cb0, r1w, wt, ooff);
                }
                if (!share_merge && bs->last_flag && tid == 0) p.counters[s] = 0;
            }
            ++piece;
            if (piece_end >= t_end || !next_piece(p, w) || w.first >= t_end) break;
            t = w.first;
        }
        // Cooperative launch: merge this block's share of each split segment
        // it worked on (only a range's first and last pieces can be split),
        // once every piece of it has arrived.  Arrivals never wait and all
        // blocks are resident, so every wait ends.  The segment counter then
        // counts the finished shares; the last one resets it.
        if (ok && share_merge) ok = sm_sync();   // both groups see walk_last
#pragma unroll 1
        for (int k = 0; k < 2 && ok && share_merge; ++k) {
            if (k == 1 && piece < 2) break;
            const Walk sw = k == 0 ? bs->walk : bs->walk_last;
            if (sw.first >= t_begin && sw.first + sw.ntiles <= t_end) continue;   // whole
            const int c0 = sw.first >= t_begin ? c : sp.owner(sw.first);
            const int c1 = sw.first + sw.ntiles <= t_end ? c : sp.owner(sw.first + sw.ntiles - 1);
            ok = share_merge_segment<D, GA, kSoftmaxThreads>(
                p, bs, reinterpret_cast<float *>(smem + C::OFF_SLOTS), sw, c0, c1, c, tid, sm_ctr, k, piece);
            if (!ok) { set_abort(bs, p); break; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (CL) {
        // A block with no tiles contributes nothing (m = -inf, l = 0).  Then
        // every block's partial is in its shared memory; block `rank` merges
        // its share of the list's rows x (D/4) float4 units from all of them
        // (running maximum over the blocks in order, as the shared merge),
        // and the cluster meets again before any block leaves.
        float *part = reinterpret_cast<float *>(smem + C::OFF_SLOTS);
        if (!has_work)
            for (int r = tid; r < p.rows; r += kThreadsTC) {
                part[p.rows * D + r] = neg_inf();
                part[p.rows * D + p.rows + r] = 0.f;
            }
        ptx::cluster_sync();
        cluster_merge<D>(p, smem_base + C::OFF_SLOTS, tid);
        ptx::cluster_sync();
    }
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
    if (AP) append_exit(p);
}

// ------------------------------------------------------------- host side
// [B, Hkv, cap, d] cache -> 4-D map (d, cap, Hkv, B); rows past the capacity
// (or before 0) read as zeros.  bf16: box (64, 128, 1, 1) with the 128-byte
// swizzle the MMA descriptors expect.  int8: rows of d / 2 pairs of codes,
// one box (64 pairs = 128 codes, 128 bytes) per 128 codes, also 128-byte
// swizzled (the widening threads read it).
inline bool make_map(CUtensorMap *m, const void *base, const int64_t *st, const Params &p,
                     cuuint32_t box_rows = TT) {
    // (int8 codes are moved as pairs: 16-bit elements, d / 2 per row)
    const int es = p.kv_int8 ? 1 : 2;
    const cuuint64_t row_elems = p.kv_int8 ? (cuuint64_t)p.d / 2 : (cuuint64_t)p.d;
    cuuint64_t dims[4] = {row_elems, (cuuint64_t)p.cap, (cuuint64_t)p.Hkv, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)(st[2] * es), (cuuint64_t)(st[1] * es),
                             (cuuint64_t)(st[0] * es)};
    cuuint32_t box[4] = {64u, box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode_cached(m, p.kv_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         4, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

// [B, n_q, Hq, d] queries -> 4-D map (d, n_q, Hq, B), box (64, n_q, g, 1):
// one box holds a segment's packed rows for 64 columns (gather: box
// (64, 1, g, 1), the g heads of one query row).
inline bool make_qmap(CUtensorMap *m, const Params &p) {
    cuuint64_t dims[4] = {(cuuint64_t)p.d, (cuuint64_t)p.n_q, (cuuint64_t)p.Hq, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)p.qs[1] * 2, (cuuint64_t)p.qs[2] * 2,
                             (cuuint64_t)p.qs[0] * 2};
    cuuint32_t box[4] = {64, p.mode == kGather ? 1u : (cuuint32_t)p.n_q, (cuuint32_t)p.g, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t *>(p.q), dims,
                         strides, box, estr, CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

// Gather: the cache seen as 2-D rows (d, Y) of stride rs elements, with rs
// the smallest of the three outer strides (each a multiple of it); gather4
// loads read one 64-column, one-row box per listed cell.
inline bool gather_rows(const Params &p, int64_t *rs, int64_t *Y, int64_t g[3]) {
    const int64_t *st = p.ks;
    if (p.vs[0] != st[0] || p.vs[1] != st[1] || p.vs[2] != st[2]) return false;
    int64_t r = st[0];
    for (int k = 1; k < 3; ++k) r = st[k] < r ? st[k] : r;
    if (r < p.d) return false;
    for (int k = 0; k < 3; ++k)
        if (st[k] % r) return false;
    g[0] = st[0] / r;
    g[1] = st[1] / r;
    g[2] = st[2] / r;
    *rs = r;
    *Y = (int64_t)(p.B - 1) * g[0] + (int64_t)(p.Hkv - 1) * g[1] + (p.cap - 1) * g[2] + 1;
    return *Y < ((int64_t)1 << 31);
}

// (int8 caches: rows of d / 2 pairs of codes, one 128-code box per gather)
inline bool make_gmap(CUtensorMap *m, const void *base, const Params &p, int64_t rs, int64_t Y) {
    const int es = p.kv_int8 ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)(p.kv_int8 ? p.d / 2 : p.d), (cuuint64_t)Y};
    cuuint64_t strides[1] = {(cuuint64_t)rs * es};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t estr[2] = {1, 1};
    return encode_cached(m, p.kv_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

// Blocks of this instantiation that can be resident at once on the current
// device (0 on error); sets the dynamic shared memory opt-in the first time.
template <int D, int N, bool I8, int NV, bool GA, bool SH, bool PG, bool AP, int MK, bool CL = false>
int resident_blocks() {
    using C = Cfg<D, N, I8, NV, GA>;
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    int per_sm = 0, sms = 0;
    if (cudaFuncSetAttribute(tc_kernel<D, N, I8, NV, GA, SH, PG, AP, MK, CL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_kernel<D, N, I8, NV, GA, SH, PG, AP, MK, CL>,
                                                      kThreadsTC, C::SMEM) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    n = per_sm * sms;
    cached[dev].store(n, std::memory_order_release);
    return n;
}

template <int D, int N, bool I8, int NV = N, bool GA = false, bool SH = false, bool PG = false,
          bool AP = false, int MK = 0, bool CL = false>
int launch_dn(const TcArgs &args, int G, cudaStream_t st) {
    using C = Cfg<D, N, I8, NV, GA>;
    const int resident = resident_blocks<D, N, I8, NV, GA, SH, PG, AP, MK, CL>();
    if (resident <= 0) return -5;
    if (CL) {
        // clusters of args.p.cl blocks, one per list (G = lists x cl); all
        // of them resident at once, or -2 (the caller then splits as usual)
        auto kern = tc_kernel<D, N, I8, NV, GA, SH, PG, AP, MK, CL>;
        const int cs = args.p.cl;
        if (cs < 2 || cs > 16 || G % cs) return -2;
        if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                          cudaSuccess)
            return -2;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)G);
        cfg.blockDim = dim3(kThreadsTC);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            return -2;
        }
        if (clusters < G / cs) return -2;
        return cudaLaunchKernelEx(&cfg, kern, args) == cudaSuccess ? 0 : -5;
    }
    if (!SH && !AP) {
        tc_kernel<D, N, I8, NV, GA, SH, PG, AP, MK, CL><<<G, kThreadsTC, C::SMEM, st>>>(args);
        return cudaGetLastError() == cudaSuccess ? 0 : -5;
    }
    // shared merges or fused append: a cooperative launch (every block
    // resident)
    if (G > resident) return -2;
    TcArgs ca = args;
    ca.p.coop = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kThreadsTC);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_kernel<D, N, I8, NV, GA, SH, PG, AP, MK, CL>, ca) == cudaSuccess ? 0 : -5;
}

}  // namespace

}  // namespace fd
