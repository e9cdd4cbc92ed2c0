// fd_tc_append.cu -- launches of the tensor-core decode kernel with a fused
// K/V append (flat bf16 caches): the launch first copies the step's new rows
// (k_new / v_new, n_new per sequence and kv head) into the caches at each
// sequence's old length, meets once at a grid-wide barrier (a cooperative
// launch: every block is resident), then attends over the prefix including
// the new rows exactly as the dense mode does; the last block to finish
// writes the new lengths.  One launch replaces the cache-write launch and
// the attention launch of a decode step.
#include "fd_tc_kernel.cuh"

namespace fd {

namespace {

template <int D>
int launch_append_d(const TcArgs &args, int G, cudaStream_t st) {
    const Params &p = args.p;
    const int rows = p.rows;
    // few segments at head_dim 256: the shared-merge kernels, as for the
    // plain dense calls
    if constexpr (D == 256) {
        if (p.nseg * 8 <= (int64_t)G && rows <= 32)
            return rows <= 16 ? launch_dn<D, 16, false, 16, false, true, false, true>(args, G, st)
                              : launch_dn<D, 32, false, 32, false, true, false, true>(args, G, st);
    }
    if (rows <= 16) return launch_dn<D, 16, false, 16, false, false, false, true>(args, G, st);
    if (rows <= 32) return launch_dn<D, 32, false, 32, false, false, false, true>(args, G, st);
    if (rows <= 48) return launch_dn<D, 48, false, 48, false, false, false, true>(args, G, st);
    if (rows <= 64) return launch_dn<D, 64, false, 64, false, false, false, true>(args, G, st);
    return -2;
}

}  // namespace

int launch_tc_append(const Params &p, int G, cudaStream_t st) {
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    if (!make_map(&args.tk, p.k, p.ks, p) || !make_map(&args.tv, p.v, p.vs, p) ||
        !make_qmap(&args.tq, p))
        return -5;
    return p.d == 128 ? launch_append_d<128>(args, G, st) : launch_append_d<256>(args, G, st);
}

}  // namespace fd
