// fd_tc_paged.cu -- launches of the tensor-core decode kernel over paged
// caches: a pool of fixed-size pages [num_pages, Hkv, page_size, d] and a
// per-sequence block table.  Everything but the row lookup is the dense
// prefix mode (segments, split, causal window, in-launch merge).  The
// producer reads a tile wholly inside the length as tiled box loads, one
// per run of rows that lies on one page (4-D map of the pool), and the
// segment's partial last tile row by row with tile::gather4 (2-D map of the
// pool's rows; rows past the length are row -1 and read as zeros), so rows
// past the length are never read.  Page sizes without such runs (not a
// multiple of 128, nor a power of two from 8 to 64) gather every tile.
#include "fd_tc_kernel.cuh"

namespace fd {

namespace {

// The pool seen as 2-D rows (d elements each, stride rs elements), with rs
// the smallest of its three outer strides (each a multiple of it, rs >= d).
// Row (page, hk, r) is page*g[0] + hk*g[1] + r*g[2]; Y rows in all.
bool paged_rows(const Params &p, int64_t *rs, int64_t *Y, int64_t g[3]) {
    const int64_t *st = p.ks;
    if (p.vs[0] != st[0] || p.vs[1] != st[1] || p.vs[2] != st[2]) return false;
    int64_t r = st[0];
    for (int k = 1; k < 3; ++k) r = st[k] < r ? st[k] : r;
    if (r < p.d) return false;
    for (int k = 0; k < 3; ++k)
        if (st[k] % r) return false;
    for (int k = 0; k < 3; ++k) g[k] = st[k] / r;
    *rs = r;
    *Y = (p.num_pages - 1) * g[0] + (int64_t)(p.Hkv - 1) * g[1] + (int64_t)(p.page_size - 1) * g[2] + 1;
    return *Y < ((int64_t)1 << 31);
}

// Rows per tiled box: a tile of 128 positions is 128 / prow runs of prow rows
// that each lie on one page (page_size a multiple of 128, or 8 .. 64 and a
// power of two); 0 where no such split exists (the tiles are then gathered).
int tiled_rows(int32_t page_size) {
    if (page_size % 128 == 0) return 128;
    if (page_size >= 8 && page_size < 128 && 128 % page_size == 0) return page_size;
    return 0;
}

// The pool as a 4-D map (d, page_size, Hkv, num_pages), box (64, prow, 1, 1),
// 128-byte swizzled like the flat caches' maps (int8: 16-bit pairs of codes).
bool make_tiled_pmap(CUtensorMap *m, const void *base, const int64_t *st, const Params &p,
                     int prow) {
    const int es = p.kv_int8 ? 1 : 2;
    const cuuint64_t row_elems = p.kv_int8 ? (cuuint64_t)p.d / 2 : (cuuint64_t)p.d;
    cuuint64_t dims[4] = {row_elems, (cuuint64_t)p.page_size, (cuuint64_t)p.Hkv,
                          (cuuint64_t)p.num_pages};
    cuuint64_t strides[3] = {(cuuint64_t)(st[2] * es), (cuuint64_t)(st[1] * es),
                             (cuuint64_t)(st[0] * es)};
    cuuint32_t box[4] = {64u, (cuuint32_t)prow, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode_cached(m, p.kv_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         4, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

// bf16 pools: rows of d elements, box (64, 1) per gather4 row; int8 pools:
// rows of d / 2 pairs of codes moved as 16-bit elements, one box per 128
// codes.  Both 128-byte swizzled, as the tiled maps of flat caches.
bool make_pmap(CUtensorMap *m, const void *base, const Params &p, int64_t rs, int64_t Y) {
    const int es = p.kv_int8 ? 1 : 2;
    const cuuint64_t row_elems = p.kv_int8 ? (cuuint64_t)p.d / 2 : (cuuint64_t)p.d;
    cuuint64_t dims[2] = {row_elems, (cuuint64_t)Y};
    cuuint64_t strides[1] = {(cuuint64_t)(rs * es)};
    cuuint32_t box[2] = {64, 1};
    cuuint32_t estr[2] = {1, 1};
    return encode_cached(m, p.kv_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supports_paged(const Params &p) {
    int64_t rs, Y, g[3];
    return p.mode == kPaged && p.page_size >= 1 && p.num_pages >= 1 && paged_rows(p, &rs, &Y, g);
}

int launch_tc_paged(const Params &p, int G, cudaStream_t st) {
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    int64_t rs, Y, g[3];
    if (!paged_rows(p, &rs, &Y, g)) return -2;
    args.gs0 = g[0];
    args.gs1 = g[1];
    args.gs2 = g[2];
    if (!make_pmap(&args.gk, p.k, p, rs, Y) || !make_pmap(&args.gv, p.v, p, rs, Y) ||
        !make_qmap(&args.tq, p))
        return -5;
    args.prow = tiled_rows(p.page_size);
    if (args.prow > 0) {
        if (!make_tiled_pmap(&args.tk, p.k, p.ks, p, args.prow) ||
            !make_tiled_pmap(&args.tv, p.v, p.vs, p, args.prow))
            return -5;
    } else {
        args.tk = args.gk;   // (unused: every tile is gathered)
        args.tv = args.gv;
    }
    const int rows = p.rows;
    if (p.kv_int8 && p.d == 128)
        return rows <= 8    ? launch_dn<128, 16, true, 8, false, false, true>(args, G, st)
               : rows <= 16 ? launch_dn<128, 16, true, 16, false, false, true>(args, G, st)
                            : launch_dn<128, 32, true, 32, false, false, true>(args, G, st);
    if (p.kv_int8)
        return rows <= 8    ? launch_dn<256, 16, true, 8, false, false, true>(args, G, st)
               : rows <= 16 ? launch_dn<256, 16, true, 16, false, false, true>(args, G, st)
                            : launch_dn<256, 32, true, 32, false, false, true>(args, G, st);
    if (p.d == 128)
        return rows <= 16   ? launch_dn<128, 16, false, 16, false, false, true>(args, G, st)
               : rows <= 32 ? launch_dn<128, 32, false, 32, false, false, true>(args, G, st)
                            : launch_dn<128, 64, false, 64, false, false, true>(args, G, st);
    return rows <= 16   ? launch_dn<256, 16, false, 16, false, false, true>(args, G, st)
           : rows <= 32 ? launch_dn<256, 32, false, 32, false, false, true>(args, G, st)
                        : launch_dn<256, 64, false, 64, false, false, true>(args, G, st);
}

}  // namespace fd
