// fd_api.cu -- the C ABI of libfd.so (declared in include/fd.h): host-side
// validation, workspace management, the thread-block count and the launch.
// Every check runs before the first CUDA call; nothing here allocates,
// frees, synchronises or reads device data during a decode call.
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>

#include "fd.h"
#include "fd_internal.h"
#include "fd_launch.h"

struct fd_workspace {
    void *base;
    size_t bytes;
    int64_t max_segments;
    int32_t max_rows, head_dim, max_ctas;
    int32_t *counters;
    int32_t *status;
    float *partials;
    size_t partial_floats;
    int device;
};

namespace {

constexpr int kVersion = 1;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s per internal wait

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
    size_t counters_off, status_off, partials_off, total;
    size_t partial_floats;
};

WsLayout ws_layout(int64_t max_segments, int32_t max_rows, int32_t head_dim,
                   int32_t max_ctas) {
    WsLayout L;
    L.counters_off = 0;
    L.status_off = align_up((size_t)max_segments * 4, 256);
    L.partials_off = L.status_off + 256;
    L.partial_floats = (size_t)(max_segments + max_ctas) *
                       (size_t)fd::slot_floats(max_rows, head_dim);
    L.total = L.partials_off + align_up(L.partial_floats * 4, 256);
    return L;
}

int sm_count_current() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

int esize(int32_t dt) {
    switch (dt) {
        case FD_BF16: return 2;
        case FD_F32: return 4;
        case FD_I8: return 1;
        case FD_I32: return 4;
        default: return 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Basic structural check of a tensor descriptor.
int check_tensor(const fd_tensor *t, int ndim) {
    if (!t || !t->data || t->ndim != ndim || esize(t->dtype) == 0) return FD_ERR_ARG;
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0 || t->stride[i] < 0) return FD_ERR_ARG;
    return FD_OK;
}

int kernel_tile(int32_t kernel) {
    return kernel == FD_KERNEL_TC ? fd::tc_tile_tokens() : fd::simt_tile_tokens();
}

// Blocks for an auto launch: one per SM for the tensor-core kernel (its
// shared-memory ring fills an SM), two per SM for the CUDA-core kernel;
// never more than the largest possible tile count.
// max_units: the most work units the launch can have for its capacity
// (tiles plus the per-segment charge), so that the block count, and with it
// the split, never depends on the capacity when the units outnumber it.
int32_t auto_ctas(int32_t kernel, int64_t max_units) {
    const int sms = sm_count_current();
    if (sms <= 0) return 0;
    int64_t g = (int64_t)sms * (kernel == FD_KERNEL_TC ? 1 : 2);
    if (max_units > 0 && g > max_units) g = max_units;
    return (int32_t)(g < 1 ? 1 : g);
}

// The kernel an auto request runs for a dense call with this cache dtype.
int32_t resolve(int32_t kernel, int32_t kv_dtype) {
    if (kernel != FD_KERNEL_AUTO) return kernel;
    return kv_dtype == FD_BF16 || kv_dtype == FD_I8 ? FD_KERNEL_TC : FD_KERNEL_SIMT;
}

// Shared validation and launch for the three entry points.
struct Call {
    const fd_tensor *q, *k, *v, *ks, *vs, *out;
    const int32_t *kv_lengths;
    const int32_t *idx;
    int32_t idx_len;
    const int32_t *block_table;   // paged mode: [B, max_pages]
    int32_t max_pages;
    int32_t n_q, causal;
    float scale;
    int mode;         // fd::Mode
    int kv_int8;
    const fd_opts *opts;
    // fused append (dense bf16 only): new rows [B, n_q, Hkv, d]; the lengths
    // array to update at the end of the launch (or null)
    const fd_tensor *k_new = nullptr, *v_new = nullptr;
    int32_t *len_update = nullptr;
    const float *bias = nullptr;   // gather: per-entry score bias (or null)
    const fd_tensor *mask = nullptr;   // masked: [B, n_q, cap] fp32
};

int run(const Call &c) {
    int rc;
    if (!c.opts) return FD_ERR_ARG;
    const fd_opts &o = *c.opts;
    if (o.reserved[0] || o.reserved[1]) return FD_ERR_ARG;
    if (o.wait_limit_us < 0 || o.wait_limit_us > 2000000) return FD_ERR_ARG;
    if (o.kernel != FD_KERNEL_AUTO && o.kernel != FD_KERNEL_SIMT && o.kernel != FD_KERNEL_TC)
        return FD_ERR_ARG;
    if (o.num_ctas < 0) return FD_ERR_ARG;
    if ((rc = check_tensor(c.q, 4)) || (rc = check_tensor(c.k, 4)) ||
        (rc = check_tensor(c.v, 4)) || (rc = check_tensor(c.out, 4)))
        return rc;
    const int kvdt = c.kv_int8 ? FD_I8 : FD_BF16;
    if (c.q->dtype != FD_BF16 || c.k->dtype != kvdt || c.v->dtype != kvdt) return FD_ERR_ARG;
    if (c.out->dtype != FD_BF16 && c.out->dtype != FD_F32) return FD_ERR_ARG;

    const bool paged = c.mode == fd::kPaged;
    const int64_t B = c.q->shape[0], n_q = c.q->shape[1], Hq = c.q->shape[2], d = c.q->shape[3];
    // paged: k / v are pools [num_pages, Hkv, page_size, d] and the logical
    // capacity is max_pages * page_size
    const int64_t Hkv = c.k->shape[1], rows_per = c.k->shape[2];
    if (paged && (!c.block_table || c.max_pages < 1 || rows_per < 1 || c.k->shape[0] < 1))
        return FD_ERR_ARG;
    const int64_t cap = paged ? (int64_t)c.max_pages * rows_per : rows_per;
    if (paged && cap >= ((int64_t)1 << 31)) return FD_ERR_UNSUPPORTED;
    if (n_q != c.n_q) return FD_ERR_ARG;
    for (int i = 0; i < 4; ++i) {
        if (c.k->shape[i] != c.v->shape[i]) return FD_ERR_ARG;
        if (c.out->shape[i] != c.q->shape[i]) return FD_ERR_ARG;
    }
    if ((!paged && c.k->shape[0] != B) || c.k->shape[3] != d) return FD_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || B > (1 << 24) || Hq > 4096 || cap > ((int64_t)1 << 40))
        return FD_ERR_ARG;
    if (Hq % Hkv != 0) return FD_ERR_ARG;
    if (d != 128 && d != 256) return FD_ERR_UNSUPPORTED;
    if (n_q < 1 || n_q > 6) return FD_ERR_UNSUPPORTED;
    const int64_t g = Hq / Hkv;
    const int64_t rows = c.mode == fd::kGather ? g : g * n_q;
    if (rows > FD_MAX_ROWS) return FD_ERR_UNSUPPORTED;
    if (c.q->stride[3] != 1 || c.k->stride[3] != 1 || c.v->stride[3] != 1 ||
        c.out->stride[3] != 1)
        return FD_ERR_ARG;
    // 16-byte aligned cache rows: base pointer and every stride.
    const int es = esize(kvdt);
    if (!aligned16(c.k->data) || !aligned16(c.v->data)) return FD_ERR_ALIGN;
    for (int i = 0; i < 3; ++i)
        if ((c.k->stride[i] * es) % 16 || (c.v->stride[i] * es) % 16) return FD_ERR_ALIGN;
    if (!isfinite(c.scale)) return FD_ERR_ARG;
    if (c.kv_int8) {
        if ((rc = check_tensor(c.ks, 3)) || (rc = check_tensor(c.vs, 3))) return rc;
        if (c.ks->dtype != FD_F32 || c.vs->dtype != FD_F32) return FD_ERR_ARG;
        const int64_t want[3] = {c.k->shape[0], Hkv, rows_per};
        for (int i = 0; i < 3; ++i)
            if (c.ks->shape[i] != want[i] || c.vs->shape[i] != want[i]) return FD_ERR_ARG;
    }
    if (c.mode != fd::kGather && !c.kv_lengths) return FD_ERR_ARG;
    if (c.mode == fd::kGather && (c.idx_len < 0 || (!c.idx && c.idx_len > 0))) return FD_ERR_ARG;
    if (c.causal != 0 && c.causal != 1) return FD_ERR_ARG;
    if (c.mode == fd::kMasked) {
        if ((rc = check_tensor(c.mask, 3))) return rc;
        if (c.mask->dtype != FD_F32 || c.kv_int8) return FD_ERR_ARG;
        if (c.mask->shape[0] != B || c.mask->shape[1] != n_q || c.mask->shape[2] != cap ||
            c.mask->stride[2] != 1)
            return FD_ERR_ARG;
        if (reinterpret_cast<uintptr_t>(c.mask->data) & 3) return FD_ERR_ALIGN;
    }
    const bool append = c.k_new != nullptr;
    if (append) {
        if (c.mode != fd::kDense || c.kv_int8) return FD_ERR_ARG;
        if ((rc = check_tensor(c.k_new, 4)) || (rc = check_tensor(c.v_new, 4))) return rc;
        if (c.k_new->dtype != FD_BF16 || c.v_new->dtype != FD_BF16) return FD_ERR_ARG;
        const int64_t want[4] = {B, n_q, Hkv, d};
        for (int i = 0; i < 4; ++i)
            if (c.k_new->shape[i] != want[i] || c.v_new->shape[i] != want[i]) return FD_ERR_ARG;
        if (c.k_new->stride[3] != 1 || c.v_new->stride[3] != 1) return FD_ERR_ARG;
        if (!aligned16(c.k_new->data) || !aligned16(c.v_new->data)) return FD_ERR_ALIGN;
        for (int i = 0; i < 3; ++i)
            if (c.k_new->stride[i] % 8 || c.v_new->stride[i] % 8) return FD_ERR_ALIGN;
    }

    fd_workspace *ws = o.ws;
    if (!ws) return FD_ERR_WORKSPACE;
    const int64_t nseg = c.mode == fd::kGather ? B * n_q * Hkv : B * Hkv;
    fd::Params p;
    memset(&p, 0, sizeof p);
    p.B = (int32_t)B; p.n_q = (int32_t)n_q; p.Hq = (int32_t)Hq; p.Hkv = (int32_t)Hkv;
    p.g = (int32_t)g; p.d = (int32_t)d; p.cap = cap; p.rows = (int32_t)rows;
    p.mode = c.mode; p.causal = c.mode != fd::kGather ? c.causal : 0;
    p.kv_int8 = c.kv_int8; p.out_f32 = c.out->dtype == FD_F32;
    p.scale_log2 = c.scale * 1.4426950408889634f;
    p.idx_len = c.idx_len; p.nseg = nseg;
    p.q = static_cast<const uint16_t *>(c.q->data);
    p.k = c.k->data; p.v = c.v->data;
    for (int i = 0; i < 4; ++i) {
        p.qs[i] = c.q->stride[i]; p.ks[i] = c.k->stride[i];
        p.vs[i] = c.v->stride[i]; p.os[i] = c.out->stride[i];
    }
    if (c.kv_int8) {
        p.k_scale = static_cast<const float *>(c.ks->data);
        p.v_scale = static_cast<const float *>(c.vs->data);
        for (int i = 0; i < 3; ++i) { p.kss[i] = c.ks->stride[i]; p.vss[i] = c.vs->stride[i]; }
    }
    p.kv_lengths = c.kv_lengths;
    p.idx = c.idx;
    p.bias = c.mode == fd::kGather ? c.bias : nullptr;
    if (c.mode == fd::kMasked) {
        p.mask = static_cast<const float *>(c.mask->data);
        p.ms[0] = c.mask->stride[0];
        p.ms[1] = c.mask->stride[1];
    }
    if (paged) {
        p.block_table = c.block_table;
        p.page_size = (int32_t)rows_per;
        p.max_pages = c.max_pages;
        p.num_pages = c.k->shape[0];
        p.page_shift = -1;
        for (int sh = 0; sh < 31; ++sh)
            if (((int64_t)1 << sh) == rows_per) p.page_shift = sh;
    }
    p.out = c.out->data;
    p.wait_ns = o.wait_limit_us > 0 ? (uint64_t)o.wait_limit_us * 1000u : kDefaultWaitNs;
    p.counters = ws->counters;
    p.status = ws->status;
    p.partials = ws->partials;
    if (append) {
        p.n_new = (int32_t)n_q;
        p.k_new = static_cast<const uint16_t *>(c.k_new->data);
        p.v_new = static_cast<const uint16_t *>(c.v_new->data);
        for (int i = 0; i < 4; ++i) { p.kns[i] = c.k_new->stride[i]; p.vns[i] = c.v_new->stride[i]; }
        p.len_update = c.len_update;
        p.grid = ws->status + 32;   // two launch counters in the status block
    }

    // Kernel choice: the tensor-core kernel serves what fd::tc_supports
    // accepts (dense bf16 and head_dim-128 int8 caches, bf16 gather over a
    // strided cache; q read through a TMA map); the CUDA-core kernel serves
    // every mode.
    const bool tc_ok = fd::tc_supports(p);
    int32_t kernel = o.kernel == FD_KERNEL_AUTO ? (tc_ok ? FD_KERNEL_TC : FD_KERNEL_SIMT) : o.kernel;
    if (kernel == FD_KERNEL_TC && !tc_ok) return FD_ERR_UNSUPPORTED;
    // Flat dense int8 caches with more than 32 rows on the tensor cores: each
    // kv head's query heads in `parts` parts of at most 32 rows, each part a
    // segment of its own (the caches are read once per part).  Under
    // FD_KERNEL_AUTO a workspace without room for the parts' segments takes
    // the CUDA-core kernel, which serves the rows in one pass.
    int32_t parts = 1;
    if (kernel == FD_KERNEL_TC && c.kv_int8 && rows > 32) {
        parts = fd::tc_int8_row_parts((int)n_q, (int)g);
        if (parts < 2) return FD_ERR_UNSUPPORTED;
        if (o.kernel == FD_KERNEL_AUTO && nseg * parts > ws->max_segments) {
            kernel = FD_KERNEL_SIMT;
            parts = 1;
        }
    }
    const int64_t nseg_l = nseg * parts, rows_l = rows / parts;   // as launched
    p.kvdiv = parts;
    const int tile = kernel_tile(kernel);
    const int32_t seg_units =
        kernel == FD_KERNEL_TC ? fd_seg_units(FD_KERNEL_TC, (int32_t)d, kvdt) : 0;
    const int64_t max_units =
        c.mode == fd::kGather ? nseg * (fd::ceil_div(c.idx_len, tile) + seg_units)
                              : nseg_l * (fd::ceil_div(cap, tile) + seg_units);
    int32_t G = o.num_ctas;
    // bf16 gather on the tensor cores with an automatic grid: when every
    // list fits one thread-block cluster of up to 16 blocks and all the
    // clusters fit the device at once, one cluster per list merges its
    // pieces through distributed shared memory (no global partials, fences
    // or counters); the list length alone decides, never the capacity.
    if (G == 0 && kernel == FD_KERNEL_TC && c.mode == fd::kGather && !c.kv_int8 && c.idx_len > 0) {
        const int64_t ntiles = fd::ceil_div(c.idx_len, tile);
        int dev = 0, sms = 0;
        if (ntiles >= 2 && ntiles <= 16 && cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            nseg * ntiles <= (int64_t)sms) {
            p.cl = (int32_t)ntiles;
            G = (int32_t)(nseg * ntiles);
        }
    }
    if (G == 0) {
        G = auto_ctas(kernel, max_units);
        if (G <= 0) return FD_ERR_CUDA;
    }
    if (nseg_l > ws->max_segments || rows > ws->max_rows || d > ws->head_dim || G > ws->max_ctas)
        return FD_ERR_WORKSPACE;
    if ((size_t)(nseg_l + G) * (size_t)fd::slot_floats(rows_l, d) > ws->partial_floats)
        return FD_ERR_WORKSPACE;
    p.tile = tile;
    p.seg_units = seg_units;
    // Masked prefix on the tensor-core kernel: where the workspace has room
    // past the split partials, a pass lists the visible chunks first and the
    // decode walks only those; otherwise each tile finds its chunks in place.
    if (kernel == FD_KERNEL_TC && c.mode == fd::kMasked && B <= 65535) {
        const size_t used = (size_t)(nseg + G) * (size_t)fd::slot_floats(rows, d);
        const size_t need = (size_t)fd::tc_mask_list_ints(B, cap);   // 0: no list
        if (need > 0 && used + need <= ws->partial_floats)
            p.mlist = reinterpret_cast<const int32_t *>(ws->partials + used);
    }

    cudaStream_t st = static_cast<cudaStream_t>(o.stream);
    rc = kernel == FD_KERNEL_TC ? fd::launch_tc(p, G, st) : fd::launch_simt(p, G, st);
    return rc == 0 ? FD_OK : (rc == -2 ? FD_ERR_UNSUPPORTED : FD_ERR_CUDA);
}

}  // namespace

extern "C" {

int fd_decode(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
              const int32_t *kv_lengths, int32_t n_q, int32_t causal, float scale,
              const fd_tensor *out, const fd_opts *opts) {
    Call c{q, k_cache, v_cache, nullptr, nullptr, out, kv_lengths, nullptr, 0, nullptr, 0,
           n_q, causal, scale, fd::kDense, 0, opts};
    return run(c);
}

int fd_decode_int8(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                   const fd_tensor *k_scale, const fd_tensor *v_scale,
                   const int32_t *kv_lengths, int32_t n_q, int32_t causal, float scale,
                   const fd_tensor *out, const fd_opts *opts) {
    Call c{q, k_cache, v_cache, k_scale, v_scale, out, kv_lengths, nullptr, 0, nullptr, 0,
           n_q, causal, scale, fd::kDense, 1, opts};
    return run(c);
}

int fd_decode_gather(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                     const int32_t *idx, int32_t idx_len, const fd_tensor *out,
                     const fd_opts *opts) {
    if (!q || !opts) return FD_ERR_ARG;
    float scale = opts->scale;
    if (scale == 0.f && q->ndim == 4 && q->shape[3] > 0) scale = 1.f / sqrtf((float)q->shape[3]);
    Call c{q, k_cache, v_cache, nullptr, nullptr, out, nullptr, idx, idx_len, nullptr, 0,
           q->ndim == 4 ? (int32_t)q->shape[1] : 0, 0, scale, fd::kGather, 0, opts};
    return run(c);
}

int fd_decode_gather_int8(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                          const fd_tensor *k_scale, const fd_tensor *v_scale, const int32_t *idx,
                          int32_t idx_len, const fd_tensor *out, const fd_opts *opts) {
    if (!q || !opts) return FD_ERR_ARG;
    float scale = opts->scale;
    if (scale == 0.f && q->ndim == 4 && q->shape[3] > 0) scale = 1.f / sqrtf((float)q->shape[3]);
    Call c{q, k_cache, v_cache, k_scale, v_scale, out, nullptr, idx, idx_len, nullptr, 0,
           q->ndim == 4 ? (int32_t)q->shape[1] : 0, 0, scale, fd::kGather, 1, opts};
    return run(c);
}

int fd_topk_blocks(const float *scores, int32_t B, int32_t n_q, int32_t n_blocks,
                   const int32_t *kv_lengths, int32_t block_size, int32_t top_k, int32_t *idx,
                   void *stream) {
    if (!scores || !kv_lengths || !idx) return FD_ERR_ARG;
    if (B < 1 || n_q < 1 || n_blocks < 1 || block_size < 1 || top_k < 1) return FD_ERR_ARG;
    if ((int64_t)B * n_q > ((int64_t)1 << 31) - 1) return FD_ERR_ARG;
    if (n_blocks > fd::kTopkMaxBlocks) return FD_ERR_UNSUPPORTED;
    if ((int64_t)n_blocks * block_size >= ((int64_t)1 << 31) ||
        (int64_t)top_k * block_size >= ((int64_t)1 << 28))
        return FD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(scores) & 3) || (reinterpret_cast<uintptr_t>(idx) & 3) ||
        (reinterpret_cast<uintptr_t>(kv_lengths) & 3))
        return FD_ERR_ALIGN;
    const int rc = fd::launch_topk(scores, B, n_q, n_blocks, kv_lengths, block_size, top_k, idx,
                                   static_cast<cudaStream_t>(stream));
    return rc == 0 ? FD_OK : (rc == -2 ? FD_ERR_UNSUPPORTED : FD_ERR_CUDA);
}

int fd_decode_gather_bias(const fd_tensor *q, const fd_tensor *k_cache,
                          const fd_tensor *v_cache, const int32_t *idx, const float *bias,
                          int32_t idx_len, const fd_tensor *out, const fd_opts *opts) {
    if (!q || !opts) return FD_ERR_ARG;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3)) return FD_ERR_ALIGN;
    float scale = opts->scale;
    if (scale == 0.f && q->ndim == 4 && q->shape[3] > 0) scale = 1.f / sqrtf((float)q->shape[3]);
    Call c{q, k_cache, v_cache, nullptr, nullptr, out, nullptr, idx, idx_len, nullptr, 0,
           q->ndim == 4 ? (int32_t)q->shape[1] : 0, 0, scale, fd::kGather, 0, opts};
    c.bias = bias;
    return run(c);
}

int fd_decode_masked(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                     const int32_t *kv_lengths, const fd_tensor *mask, int32_t n_q,
                     int32_t causal, float scale, const fd_tensor *out, const fd_opts *opts) {
    if (!mask) return FD_ERR_ARG;
    Call c{q, k_cache, v_cache, nullptr, nullptr, out, kv_lengths, nullptr, 0, nullptr, 0,
           n_q, causal, scale, fd::kMasked, 0, opts};
    c.mask = mask;
    return run(c);
}

int fd_decode_append(const fd_tensor *q, const fd_tensor *k_cache, const fd_tensor *v_cache,
                     const fd_tensor *k_new, const fd_tensor *v_new, int32_t *kv_lengths,
                     int32_t update_lengths, int32_t causal, float scale, const fd_tensor *out,
                     const fd_opts *opts) {
    if (!q || !k_new || !v_new) return FD_ERR_ARG;
    if (update_lengths != 0 && update_lengths != 1) return FD_ERR_ARG;
    Call c{q, k_cache, v_cache, nullptr, nullptr, out, kv_lengths, nullptr, 0, nullptr, 0,
           q->ndim == 4 ? (int32_t)q->shape[1] : 0, causal, scale, fd::kDense, 0, opts};
    c.k_new = k_new;
    c.v_new = v_new;
    c.len_update = update_lengths ? kv_lengths : nullptr;
    return run(c);
}

int fd_decode_paged(const fd_tensor *q, const fd_tensor *k_pages, const fd_tensor *v_pages,
                    const fd_tensor *k_scale, const fd_tensor *v_scale,
                    const int32_t *block_table, int32_t max_pages, const int32_t *kv_lengths,
                    int32_t n_q, int32_t causal, float scale, const fd_tensor *out,
                    const fd_opts *opts) {
    if (!k_pages) return FD_ERR_ARG;
    const int int8 = k_pages->dtype == FD_I8;
    if (!int8 && (k_scale || v_scale)) return FD_ERR_ARG;
    Call c{q, k_pages, v_pages, k_scale, v_scale, out, kv_lengths, nullptr, 0, block_table,
           max_pages, n_q, causal, scale, fd::kPaged, int8, opts};
    return run(c);
}

size_t fd_workspace_bytes(int64_t max_segments, int32_t max_rows, int32_t head_dim,
                          int32_t max_ctas) {
    if (max_segments < 1 || max_rows < 1 || head_dim < 1 || max_ctas < 1) return 0;
    return ws_layout(max_segments, max_rows, head_dim, max_ctas).total;
}

int fd_workspace_create(int64_t max_segments, int32_t max_rows, int32_t head_dim,
                        int32_t max_ctas, void *stream, fd_workspace **out) {
    if (!out || max_segments < 1 || max_rows < 1 || max_rows > FD_MAX_ROWS ||
        head_dim < 1 || head_dim > 256 || max_ctas < 1)
        return FD_ERR_ARG;
    *out = nullptr;
    const WsLayout L = ws_layout(max_segments, max_rows, head_dim, max_ctas);
    fd_workspace *ws = new (std::nothrow) fd_workspace;
    if (!ws) return FD_ERR_ARG;
    void *base = nullptr;
    if (cudaMalloc(&base, L.total) != cudaSuccess) {
        delete ws;
        return FD_ERR_CUDA;
    }
    ws->base = base;
    ws->bytes = L.total;
    ws->max_segments = max_segments;
    ws->max_rows = max_rows;
    ws->head_dim = head_dim;
    ws->max_ctas = max_ctas;
    ws->counters = reinterpret_cast<int32_t *>(static_cast<char *>(base) + L.counters_off);
    ws->status = reinterpret_cast<int32_t *>(static_cast<char *>(base) + L.status_off);
    ws->partials = reinterpret_cast<float *>(static_cast<char *>(base) + L.partials_off);
    ws->partial_floats = L.partial_floats;
    cudaGetDevice(&ws->device);
    if (cudaMemsetAsync(base, 0, L.partials_off, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaFree(base);
        delete ws;
        return FD_ERR_CUDA;
    }
    *out = ws;
    return FD_OK;
}

int fd_workspace_reset(fd_workspace *ws, void *stream) {
    if (!ws) return FD_ERR_ARG;
    const size_t n = reinterpret_cast<char *>(ws->partials) - static_cast<char *>(ws->base);
    return cudaMemsetAsync(ws->base, 0, n, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FD_OK : FD_ERR_CUDA;
}

}  // extern "C"

namespace {
__global__ void fill_i32(int32_t *p, int64_t n, int32_t value) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = value;
}
}  // namespace

extern "C" {

int fd_workspace_fill_counters(fd_workspace *ws, int32_t value, void *stream) {
    if (!ws) return FD_ERR_ARG;
    const int64_t n = ws->max_segments;
    const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    fill_i32<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(ws->counters, n, value);
    return cudaGetLastError() == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

int fd_workspace_destroy(fd_workspace *ws) {
    if (!ws) return FD_ERR_ARG;
    const cudaError_t e = cudaFree(ws->base);
    delete ws;
    return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

int fd_get_device_status(fd_workspace *ws, int32_t *status) {
    if (!ws || !status) return FD_ERR_ARG;
    return cudaMemcpy(status, ws->status, sizeof(int32_t), cudaMemcpyDeviceToHost) == cudaSuccess
               ? FD_OK : FD_ERR_CUDA;
}

int fd_get_device_diagnostics(fd_workspace *ws, int32_t *words) {
    if (!ws || !words) return FD_ERR_ARG;
    return cudaMemcpy(words, ws->status, 13 * sizeof(int32_t), cudaMemcpyDeviceToHost) == cudaSuccess
               ? FD_OK : FD_ERR_CUDA;
}

int32_t fd_auto_num_ctas(int32_t kernel, int32_t head_dim, int32_t kv_dtype, int32_t rows,
                         int64_t max_units) {
    (void)head_dim; (void)kv_dtype; (void)rows;
    return auto_ctas(resolve(kernel, kv_dtype), max_units);
}

size_t fd_masked_list_bytes(int64_t B, int64_t cap) {
    if (B < 1 || B > 65535 || cap < 1 || cap > ((int64_t)1 << 23)) return 0;
    return (size_t)fd::tc_mask_list_ints(B, cap) * 4;
}

int32_t fd_tile_tokens(int32_t kernel, int32_t head_dim, int32_t kv_dtype) {
    (void)head_dim;
    return kernel_tile(resolve(kernel, kv_dtype));
}

int64_t fd_plan(const int64_t *seg_len, int64_t nseg, int32_t tile_tokens, int32_t num_ctas,
                int32_t seg_units, int32_t *first_cta, int32_t *n_pieces) {
    if (!seg_len || nseg < 0 || tile_tokens < 1 || num_ctas < 1 || seg_units < 0 ||
        !first_cta || !n_pieces)
        return FD_ERR_ARG;
    int64_t total = 0;
    for (int64_t s = 0; s < nseg; ++s) {
        if (seg_len[s] < 0) return FD_ERR_ARG;
        const int64_t n = fd::ceil_div(seg_len[s], tile_tokens);
        total += n > 0 ? n + seg_units : 0;
    }
    const fd::Split sp{total, fd::working_blocks(total, num_ctas)};
    int64_t first = 0;   // unit index where segment s starts
    for (int64_t s = 0; s < nseg; ++s) {
        const int64_t n = fd::ceil_div(seg_len[s], tile_tokens);
        if (n == 0) {
            first_cta[s] = (int32_t)(s % num_ctas);   // block that zeroes it
            n_pieces[s] = 0;
        } else {
            // blocks whose ranges hold the segment's tiles (its units after
            // the first seg_units)
            const int32_t a = sp.owner(first + seg_units), b = sp.owner(first + seg_units + n - 1);
            first_cta[s] = a;
            n_pieces[s] = b - a + 1;
            first += n + seg_units;
        }
    }
    return total;
}

int32_t fd_seg_units(int32_t kernel, int32_t head_dim, int32_t kv_dtype) {
    if (kernel != FD_KERNEL_TC || (head_dim != 128 && head_dim != 256)) return 0;
    fd::Params p;
    memset(&p, 0, sizeof p);
    p.d = head_dim;
    p.kv_int8 = kv_dtype == FD_I8;
    return fd::tc_seg_units(p);
}

const char *fd_status_string(int status) {
    switch (status) {
        case FD_OK: return "ok";
        case FD_ERR_ARG: return "invalid argument";
        case FD_ERR_UNSUPPORTED: return "unsupported head_dim, query rows or group size";
        case FD_ERR_ALIGN: return "cache pointer or stride not 16-byte aligned";
        case FD_ERR_WORKSPACE: return "missing or too small workspace";
        case FD_ERR_CUDA: return "CUDA runtime error";
        case FD_ERR_SCRATCH: return "problem exceeds the fixed scratch of fd_decode_noalloc";
        default: return "unknown status";
    }
}

int32_t fd_version(void) { return kVersion; }

}  // extern "C"
