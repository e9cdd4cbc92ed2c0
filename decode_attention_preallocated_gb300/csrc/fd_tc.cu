// fd_tc.cu -- launches of the tensor-core decode kernel (fd_tc_kernel.cuh)
// over flat bf16 caches ([B, Hkv, cap, d]) and in index-gather mode, and the
// kernel-choice queries of the C ABI layer.  Flat int8 caches are launched
// from fd_tc_int8.cu, paged caches from fd_tc_paged.cu, fused appends from
// fd_tc_append.cu, the masked prefix from fd_tc_masked.cu (chunks found in
// place) and fd_tc_masked_list.cu (a chunk list first).
#include "fd_tc_kernel.cuh"

namespace fd {

namespace {

template <int D>
int launch_d(const TcArgs &args, int G, cudaStream_t st) {
    const int rows = args.p.rows;
    // Launches of few segments at head_dim 256 take the shared-merge kernels
    // (when the grid fits on the device at once); inside, a short launch
    // (a few tiles per block) shares its merges and a long one keeps the
    // last-arriver merge.  The choice depends on shapes only, never on the
    // capacity.
    const Params &p = args.p;
    if (D == 256 && p.nseg * 8 <= (int64_t)G) {
        if (rows <= 16 && G <= resident_blocks<D, 16, false, 16, false, true, false, false, false>())
            return launch_dn<D, 16, false, 16, false, true>(args, G, st);
        if (rows > 16 && rows <= 32 && G <= resident_blocks<D, 32, false, 32, false, true, false, false, false>())
            return launch_dn<D, 32, false, 32, false, true>(args, G, st);
    }
    if (rows <= 16) return launch_dn<D, 16, false>(args, G, st);
    if (rows <= 32) return launch_dn<D, 32, false>(args, G, st);
    if (rows <= 48) return launch_dn<D, 48, false>(args, G, st);
    if (rows <= 64) return launch_dn<D, 64, false>(args, G, st);
    return -2;
}

}  // namespace

int tc_tile_tokens() { return TT; }

// Work units charged per segment start: about the cost of a piece boundary
// (epilogue of one piece, restart of the pipeline on the next) in tile times.
// A tile of head_dim 256 streams twice the bytes of one of head_dim 128.
// int8 tiles (codes and scales) stream about half the bytes of bf16 ones.
int tc_seg_units(const Params &p) { return p.kv_int8 ? 14 : (p.d == 256 ? 6 : 9); }

int tc_int8_row_parts(int n_q, int g) {
    for (int k = 1; k <= g; ++k)
        if (g % k == 0 && (int64_t)n_q * (g / k) <= 32) return k;
    return 0;
}

bool tc_supports(const Params &p) {
    // Q goes through a tensor map: 16-byte aligned base and strides.
    const bool q_aligned = (reinterpret_cast<uintptr_t>(p.q) & 15) == 0 && p.qs[0] % 8 == 0 &&
                           p.qs[1] % 8 == 0 && p.qs[2] % 8 == 0;
    // int8 caches: head_dim 128 or 256 and up to 32 rows (one softmax
    // warpgroup; the other four warps widen the codes); flat dense launches
    // with more rows run in parts of a kv head's query heads.
    const bool int8_rows =
        p.rows <= 32 || (p.mode == kDense && p.n_new == 0 && tc_int8_row_parts(p.n_q, p.g) > 0);
    const bool shape = p.kv_int8 ? ((p.d == 128 || p.d == 256) && int8_rows)
                                 : ((p.d == 128 || p.d == 256) && p.rows <= 64);
    // gather: bf16 caches whose rows form one strided 2-D array; paged: pools
    // whose rows do (fd_tc_paged.cu)
    int64_t rs, Y, g[3];
    const bool mode = p.mode == kDense || (p.mode == kMasked && !p.kv_int8) ||
                      (p.mode == kGather && gather_rows(p, &rs, &Y, g)) ||
                      tc_supports_paged(p);
    // fused append: flat bf16 caches (fd_tc_append.cu)
    const bool append = p.n_new == 0 || (p.mode == kDense && !p.kv_int8);
    return mode && shape && append && p.rows >= 1 && p.cap < (int64_t)1 << 31 &&
           p.B < (1 << 30) && p.Hkv < (1 << 30) && q_aligned;
}

int launch_tc(const Params &p, int G, cudaStream_t st) {
    if (!tc_supports(p)) return -2;
    if (p.mode == kPaged) return launch_tc_paged(p, G, st);
    if (p.n_new > 0) return launch_tc_append(p, G, st);
    if (p.kv_int8) return launch_tc_int8(p, G, st);   // flat int8: dense or gather
    if (p.mode == kMasked) return p.mlist ? launch_tc_masked_list(p, G, st) : launch_tc_masked(p, G, st);
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    if (p.mode == kGather) {
        int64_t rs = 0, Y = 0, g[3] = {0, 0, 0};
        if (!gather_rows(p, &rs, &Y, g)) return -2;
        args.gs0 = g[0];
        args.gs1 = g[1];
        args.gs2 = g[2];
        if (!make_gmap(&args.tk, p.k, p, rs, Y) || !make_gmap(&args.tv, p.v, p, rs, Y) ||
            !make_qmap(&args.tq, p))
            return -5;
        const int rows = p.rows;
        if (p.cl > 1) {
            // one cluster of p.cl blocks per list, merging through
            // distributed shared memory; -2 (the clusters do not all fit at
            // once): the same grid splits as usual
            const int rc =
                p.d == 128 ? (rows <= 16   ? launch_dn<128, 16, false, 16, true, false, false, false, 0, true>(args, G, st)
                              : rows <= 32 ? launch_dn<128, 32, false, 32, true, false, false, false, 0, true>(args, G, st)
                                           : launch_dn<128, 64, false, 64, true, false, false, false, 0, true>(args, G, st))
                           : (rows <= 16   ? launch_dn<256, 16, false, 16, true, false, false, false, 0, true>(args, G, st)
                              : rows <= 32 ? launch_dn<256, 32, false, 32, true, false, false, false, 0, true>(args, G, st)
                                           : launch_dn<256, 64, false, 64, true, false, false, false, 0, true>(args, G, st));
            if (rc != -2) return rc;
            args.p.cl = 0;
        }
        if (p.d == 128)
            return rows <= 16   ? launch_dn<128, 16, false, 16, true>(args, G, st)
                   : rows <= 32 ? launch_dn<128, 32, false, 32, true>(args, G, st)
                                : launch_dn<128, 64, false, 64, true>(args, G, st);
        return rows <= 16   ? launch_dn<256, 16, false, 16, true>(args, G, st)
               : rows <= 32 ? launch_dn<256, 32, false, 32, true>(args, G, st)
                            : launch_dn<256, 64, false, 64, true>(args, G, st);
    }
    if (!make_map(&args.tk, p.k, p.ks, p) || !make_map(&args.tv, p.v, p.vs, p) ||
        !make_qmap(&args.tq, p))
        return -5;
    if (p.d == 128) return launch_d<128>(args, G, st);
    return launch_d<256>(args, G, st);
}

}  // namespace fd
