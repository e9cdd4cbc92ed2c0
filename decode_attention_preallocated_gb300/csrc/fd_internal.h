// fd_internal.h -- launch parameters and the split-KV partitioner, shared by
// the host launcher and the kernels (plain C++, usable from host and device).
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define FD_HD __host__ __device__ __forceinline__
#else
#define FD_HD inline
#endif

namespace fd {

// kPaged: the dense prefix mode over a paged cache (a pool of fixed-size
// pages and a per-sequence block table); it shares the dense mode's segments,
// tiles and masks and differs only in where a position's row lives.
// kMasked: the dense prefix mode with an additive per-(query row, position)
// mask; the CUDA-core kernel skips tiles in which the mask leaves nothing
// visible.
enum Mode : int32_t { kDense = 0, kGather = 1, kPaged = 2, kMasked = 3 };

// Everything a kernel needs, passed by value as one __grid_constant__ block.
struct Params {
    // problem
    int32_t B, n_q, Hq, Hkv, g, d;
    int64_t cap;
    int32_t rows;          // query rows per segment: g*n_q (dense) or g (gather)
    int32_t mode;          // Mode
    int32_t causal;
    int32_t kv_int8;
    int32_t out_f32;
    int32_t tile;          // cache positions per tile
    int32_t seg_units;     // extra work units the split charges at the start of
                           // each non-empty segment (0: plain tile split)
    int32_t coop;          // tensor-core kernel launched cooperatively (all
                           // blocks resident): split segments may share merges
    uint64_t wait_ns;      // tensor-core kernel: bound on each internal wait (ns);
                           // one that runs out sets FD_DEV_INTERNAL
    float scale_log2;      // scale * log2(e): scores are kept in the log2 domain
    int32_t idx_len;
    int64_t nseg;          // segments: B*Hkv (dense) or B*n_q*Hkv (gather)
    // tensors (strides in elements)
    const uint16_t *q;     int64_t qs[4];
    const void *k;         int64_t ks[4];
    const void *v;         int64_t vs[4];
    const float *k_scale;  int64_t kss[3];
    const float *v_scale;  int64_t vss[3];
    const int32_t *kv_lengths;
    const int32_t *idx;
    const float *bias;     // gather: optional [B, n_q, idx_len] fp32 added to each
                           // entry's score (-inf drops the entry)
    const float *mask;     // masked: [B, n_q, cap] fp32 added to the scores
    int64_t ms[2];         //   (strides of B and n_q; positions contiguous)
    // masked, tensor-core kernel: the visible 32-position chunks of each
    // sequence in ascending order (row b starts at b * mls) and their count
    // per sequence, written by the chunk-list pass before the decode launch;
    // the decode then walks ceil(count / 4) tiles of four listed chunks.
    // Null: each tile of the prefix finds its visible chunks in place.
    const int32_t *mlist;
    const int32_t *mcnt;
    int64_t mls;
    // gather, tensor-core kernel: when > 1, each list is one thread-block
    // cluster of `cl` blocks (a share of its tiles each) whose partials merge
    // through distributed shared memory; 0 otherwise
    int32_t cl;
    // flat int8 caches, tensor-core kernel, more than 32 rows: each kv head's
    // query heads are served in `kvdiv` parts of g / kvdiv heads (at most 32
    // rows each), as if there were Hkv * kvdiv kv heads: Hkv, g, rows and
    // nseg then describe the parts, and kv head hk of a part reads the
    // caches' kv head hk / kvdiv; 0 or 1 otherwise
    int32_t kvdiv;
    // paged caches: logical position j of sequence b lives at row j % page_size
    // of pool page block_table[b * max_pages + j / page_size]; the caches'
    // strides are then (page, kv head, row in page); cap = max_pages * page_size
    const int32_t *block_table;
    int32_t page_size, max_pages;
    int32_t page_shift;    // log2(page_size) when it is a power of two, else -1
    int64_t num_pages;
    // fused append (flat bf16 caches): n_new rows per (sequence, kv head),
    // k_new / v_new [B, n_new, Hkv, d], are written at positions
    // base_b .. base_b + n_new - 1 with base_b = kv_lengths[b] (clamped to
    // [0, cap]) and attended as part of the prefix, whose length is then
    // min(base_b + n_new, cap); len_update (non-null) receives that length
    // when the launch ends.  n_new = 0 otherwise.
    int32_t n_new;
    const uint16_t *k_new; int64_t kns[4];
    const uint16_t *v_new; int64_t vns[4];
    int32_t *len_update;
    int32_t *grid;         // [2] launch counters in the workspace (barrier,
                           // exit), zero between launches
    void *out;             int64_t os[4];
    // workspace
    int32_t *counters;     // [nseg], zero between launches
    int32_t *status;       // sticky FD_DEV_* bits
    float *partials;       // [(nseg + num_ctas - 1) * slot_floats(rows, d)]
};

// Balanced split of `total` tiles over G thread blocks: block c takes tiles
// [start(c), start(c+1)).  A (sequence, kv head) segment whose tiles straddle
// block boundaries is shared by several blocks ("pieces"); piece (s, c) uses
// workspace slot s + c, which is unique because block ranges are ordered the
// same way as segments.
struct Split {
    int64_t total;
    int32_t G;
    FD_HD int64_t start(int32_t c) const { return (int64_t)c * total / G; }
    // The block whose range holds tile t (0 <= t < total).
    FD_HD int32_t owner(int64_t t) const {
        return (int32_t)(((t + 1) * (int64_t)G + total - 1) / total - 1);
    }
};

FD_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Floats in one workspace slot: O[rows][d], then m[rows] and l[rows], padded
// so that every slot starts on a 16-byte boundary.
FD_HD int64_t slot_floats(int64_t rows, int64_t d) {
    return rows * d + ((2 * rows + 3) / 4) * 4;
}

// Blocks that get work: never more than there are tiles, so every working
// block owns at least one tile and the blocks sharing a segment are
// consecutive.
FD_HD int32_t working_blocks(int64_t total, int32_t grid) {
    return total < (int64_t)grid ? (int32_t)total : grid;
}

// Length of sequence b after clamping to [0, cap].
FD_HD int64_t clamp_len(int64_t L, int64_t cap) {
    return L < 0 ? 0 : (L > cap ? cap : L);
}

}  // namespace fd
