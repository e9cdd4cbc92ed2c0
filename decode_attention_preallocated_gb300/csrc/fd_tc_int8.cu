// fd_tc_int8.cu -- launches of the tensor-core decode kernel over flat int8
// caches (head_dim 128 or 256, up to 32 rows; the dense prefix with more rows
// in parts of each kv head's query heads), dense prefix and index gather, in
// a translation unit of their own.
#include "fd_tc_kernel.cuh"

namespace fd {

int launch_tc_int8(const Params &p, int G, cudaStream_t st) {
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    const int rows = p.rows;
    if (p.mode == kGather) {
        // the listed cells' codes fetched row by row (tile::gather4) from the
        // caches seen as 2-D arrays of rows
        int64_t rs = 0, Y = 0, g[3] = {0, 0, 0};
        if (!gather_rows(p, &rs, &Y, g)) return -2;
        args.gs0 = g[0];
        args.gs1 = g[1];
        args.gs2 = g[2];
        if (!make_gmap(&args.tk, p.k, p, rs, Y) || !make_gmap(&args.tv, p.v, p, rs, Y) ||
            !make_qmap(&args.tq, p))
            return -5;
        if (p.d == 128)
            return rows <= 8    ? launch_dn<128, 16, true, 8, true>(args, G, st)
                   : rows <= 16 ? launch_dn<128, 16, true, 16, true>(args, G, st)
                                : launch_dn<128, 32, true, 32, true>(args, G, st);
        return rows <= 8    ? launch_dn<256, 16, true, 8, true>(args, G, st)
               : rows <= 16 ? launch_dn<256, 16, true, 16, true>(args, G, st)
                            : launch_dn<256, 32, true, 32, true>(args, G, st);
    }
    if (!make_map(&args.tk, p.k, p.ks, p) || !make_map(&args.tv, p.v, p.vs, p)) return -5;
    if (p.kvdiv > 1) {
        // more than 32 rows: kv head hk's query heads in kvdiv parts of
        // g / kvdiv heads, each part a segment of its own (as kv head
        // hk * kvdiv + part, whose caches are kv head hk's); the maps of the
        // caches above keep the real kv heads, the map of q takes a part's
        // heads per box
        const int k = p.kvdiv;
        if (p.g % k || p.rows % k || p.rows / k > 32) return -2;
        args.p.Hkv = p.Hkv * k;
        args.p.g = p.g / k;
        args.p.rows = p.rows / k;
        args.p.nseg = p.nseg * k;
    }
    if (!make_qmap(&args.tq, args.p)) return -5;
    const int rows_part = args.p.rows;
    if (p.d == 128)
        return rows_part <= 8    ? launch_dn<128, 16, true, 8>(args, G, st)
               : rows_part <= 16 ? launch_dn<128, 16, true>(args, G, st)
                                 : launch_dn<128, 32, true>(args, G, st);
    return rows_part <= 8    ? launch_dn<256, 16, true, 8>(args, G, st)
           : rows_part <= 16 ? launch_dn<256, 16, true>(args, G, st)
                             : launch_dn<256, 32, true>(args, G, st);
}

}  // namespace fd
