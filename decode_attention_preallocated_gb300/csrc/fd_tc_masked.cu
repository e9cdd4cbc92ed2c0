// fd_tc_masked.cu -- launches of the tensor-core decode kernel for the masked
// prefix: the dense prefix (optionally causal) over flat bf16 caches with an
// additive fp32 mask [B, n_q, cap] ("qwen4exp : gather-based sparse attention
// for QSA decode", llama.cpp #28213: the selection as a mask over the window;
// its Metal kernel skips the chunks the mask hides).  The caches' maps load 32
// rows per box; the producer requests only the 32-position chunks of a tile
// that some query row sees, so hidden chunks cost no memory traffic and no
// copy; the slots start zeroed and a hidden chunk keeps older, finite rows of
// the filled prefix, whose scores the softmax masks.
#include "fd_tc_kernel.cuh"

namespace fd {

int launch_tc_masked(const Params &p, int G, cudaStream_t st) {
    TcArgs args;
    memset(&args, 0, sizeof args);
    args.p = p;
    // 32-row boxes (one chunk) and 128-row boxes (four consecutive chunks)
    if (!make_map(&args.tk, p.k, p.ks, p, 32) || !make_map(&args.tv, p.v, p.vs, p, 32) ||
        !make_map(&args.gk, p.k, p.ks, p) || !make_map(&args.gv, p.v, p.vs, p) ||
        !make_qmap(&args.tq, p))
        return -5;
    const int rows = p.rows;
    if (p.d == 128)
        return rows <= 16   ? launch_dn<128, 16, false, 16, false, false, false, false, true>(args, G, st)
               : rows <= 32 ? launch_dn<128, 32, false, 32, false, false, false, false, true>(args, G, st)
               : rows <= 48 ? launch_dn<128, 48, false, 48, false, false, false, false, true>(args, G, st)
                            : launch_dn<128, 64, false, 64, false, false, false, false, true>(args, G, st);
    return rows <= 16   ? launch_dn<256, 16, false, 16, false, false, false, false, true>(args, G, st)
           : rows <= 32 ? launch_dn<256, 32, false, 32, false, false, false, false, true>(args, G, st)
           : rows <= 48 ? launch_dn<256, 48, false, 48, false, false, false, false, true>(args, G, st)
                        : launch_dn<256, 64, false, 64, false, false, false, false, true>(args, G, st);
}

}  // namespace fd
