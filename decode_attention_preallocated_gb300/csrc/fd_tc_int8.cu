// fd_tc_int8.cu -- launches of the tensor-core decode kernel over flat int8
// caches (head_dim 128, up to 32 rows), in a translation unit of their own.
#include "fd_tc_kernel.cuh"

namespace fd {

int launch_tc_int8(const Params &p, int G, cudaStream_t st) {
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    if (!make_map(&args.tk, p.k, p.ks, p) || !make_map(&args.tv, p.v, p.vs, p) ||
        !make_qmap(&args.tq, p))
        return -5;
    const int rows = p.rows;
    return rows <= 8    ? launch_dn<128, 16, true, 8>(args, G, st)
           : rows <= 16 ? launch_dn<128, 16, true>(args, G, st)
                        : launch_dn<128, 32, true>(args, G, st);
}

}  // namespace fd
