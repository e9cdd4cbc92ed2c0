// fd_noalloc.cu -- fd_decode_noalloc: dense prefix decode that allocates
// nothing.
//
// Some callers cannot call cudaMalloc at all: a host application whose own
// allocator owns every byte of device memory, a process that runs under a
// hard device-memory cap, or a plugin loaded into an engine that forbids
// allocation after start-up.  fd_decode needs a workspace made by
// fd_workspace_create (which calls cudaMalloc); this entry point instead
// keeps that scratch -- the split partials, one completion counter per
// (sequence, kv head) and the status word -- in the fixed-size array below,
// which the CUDA runtime places in device memory when the library's module
// is loaded on a device.
//
// Limits and sharing:
//   * kScratchBytes (8 MiB) per device that loads the library, held until
//     the process exits; at most kMaxSegments (sequence, kv head) pairs, and
//     the thread-block count is reduced so the split partials fit.  A
//     problem whose partials cannot fit even with one block per segment is
//     rejected with FD_ERR_SCRATCH before anything is launched.
//   * Every call uses the same array.  Each call first clears the counters
//     and the status word on its stream (cudaMemsetAsync, no allocation), so
//     stale contents of an earlier call never matter; calls that overlap on
//     the GPU (different streams, or different host threads without
//     ordering) race on the array and must not be issued.
//   * Host code never sees the array's device address through its name, so
//     every call that is not being captured looks the address up again
//     (cudaGetSymbolAddress, with the caller's device current) and keeps it
//     for that device; a call made while its stream is being captured uses
//     the address kept by the last uncaptured call on the device.  The first
//     call on a device (and the first after a device reset, or in another
//     context) must therefore come before any stream capture.
//   * The status word exists because the kernel writes it (a length outside
//     [0, cap] is clamped and flagged, as in fd_decode); this entry point
//     does not report it.
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "fd.h"
#include "fd_internal.h"
#include "fd_launch.h"

namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;
constexpr int64_t kMaxSegments = 4096;
constexpr size_t kStatusOff = (size_t)kMaxSegments * 4;   // counters first
constexpr size_t kPartialsOff = kStatusOff + 256;         // then status, padded
constexpr size_t kPartialFloats = (kScratchBytes - kPartialsOff) / 4;

static __device__ __align__(256) unsigned char g_fd_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};

// Device address of g_fd_scratch on the current device (host code only ever
// sees a stand-in for the array's name, never its device address).  Looked
// up on every call whose stream is not being captured, so a device reset or
// another context made current is picked up; a captured call takes the
// address the last uncaptured call on this device found.
int scratch_on_current_device(cudaStream_t st, void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FD_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return FD_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fd_scratch) != cudaSuccess || !p) return FD_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    if (!g_scratch_addr[dev]) return FD_ERR_CUDA;   // first call inside a capture
    *out = g_scratch_addr[dev];
    return FD_OK;
}

bool valid4(const fd_tensor *t, int32_t dtype) {
    if (!t || !t->data || t->ndim != 4 || t->dtype != dtype) return false;
    for (int i = 0; i < 4; ++i)
        if (t->shape[i] < 0 || t->stride[i] < 0) return false;
    return t->stride[3] == 1;
}

}  // namespace

extern "C" int fd_decode_noalloc(const fd_tensor *q, const fd_tensor *k_cache,
                                 const fd_tensor *v_cache, const int32_t *kv_lengths,
                                 int32_t n_q, int32_t causal, float scale,
                                 const fd_tensor *out, void *stream, int32_t num_ctas) {
    if (!valid4(q, FD_BF16) || !valid4(k_cache, FD_BF16) || !valid4(v_cache, FD_BF16) || !out ||
        !valid4(out, out->dtype) || (out->dtype != FD_BF16 && out->dtype != FD_F32) ||
        !kv_lengths || (causal != 0 && causal != 1) || num_ctas < 0 || !isfinite(scale))
        return FD_ERR_ARG;
    const int64_t B = q->shape[0], Hq = q->shape[2], d = q->shape[3];
    const int64_t Hkv = k_cache->shape[1], cap = k_cache->shape[2];
    if (q->shape[1] != n_q) return FD_ERR_ARG;
    for (int i = 0; i < 4; ++i)
        if (k_cache->shape[i] != v_cache->shape[i] || out->shape[i] != q->shape[i])
            return FD_ERR_ARG;
    if (k_cache->shape[0] != B || k_cache->shape[3] != d || B < 1 || Hq < 1 || Hkv < 1 ||
        Hq % Hkv != 0 || B > (1 << 24) || cap > ((int64_t)1 << 40))
        return FD_ERR_ARG;
    if ((d != 128 && d != 256) || n_q < 1 || n_q > 6) return FD_ERR_UNSUPPORTED;
    const int64_t g = Hq / Hkv, rows = g * n_q;
    if (rows > FD_MAX_ROWS) return FD_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k_cache->data) & 15) ||
        (reinterpret_cast<uintptr_t>(v_cache->data) & 15))
        return FD_ERR_ALIGN;
    for (int i = 0; i < 3; ++i)
        if ((k_cache->stride[i] * 2) % 16 || (v_cache->stride[i] * 2) % 16) return FD_ERR_ALIGN;

    // Size check against the fixed scratch: one slot per segment plus one per
    // block; fewer blocks when the partials would not fit.
    const int64_t nseg = B * Hkv;
    const int64_t slot = fd::slot_floats(rows, d);
    if (nseg > kMaxSegments || (nseg + 1) * slot > (int64_t)kPartialFloats) return FD_ERR_SCRATCH;
    const int tile = fd::simt_tile_tokens();
    int64_t G = num_ctas;
    if (G == 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FD_ERR_CUDA;
        G = 2 * (int64_t)sms;
        const int64_t max_tiles = nseg * fd::ceil_div(cap, tile);
        if (max_tiles > 0 && G > max_tiles) G = max_tiles;
        if (G < 1) G = 1;
    }
    const int64_t fit = (int64_t)kPartialFloats / slot - nseg;
    if (G > fit) {
        if (num_ctas > 0) return FD_ERR_SCRATCH;   // an explicit count that does not fit
        G = fit;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    int rc = scratch_on_current_device(st, &scratch);
    if (rc != FD_OK) return rc;
    // Counters and status must start at zero; the array keeps the last call's
    // contents, so clear them on this call's stream first.
    if (cudaMemsetAsync(scratch, 0, kPartialsOff, st) != cudaSuccess) return FD_ERR_CUDA;

    fd::Params p;
    memset(&p, 0, sizeof p);
    p.B = (int32_t)B; p.n_q = n_q; p.Hq = (int32_t)Hq; p.Hkv = (int32_t)Hkv;
    p.g = (int32_t)g; p.d = (int32_t)d; p.cap = cap; p.rows = (int32_t)rows;
    p.mode = fd::kDense; p.causal = causal; p.kv_int8 = 0;
    p.out_f32 = out->dtype == FD_F32; p.tile = tile;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_ns = 2000000000ull;
    p.nseg = nseg;
    p.q = static_cast<const uint16_t *>(q->data);
    p.k = k_cache->data; p.v = v_cache->data;
    for (int i = 0; i < 4; ++i) {
        p.qs[i] = q->stride[i]; p.ks[i] = k_cache->stride[i];
        p.vs[i] = v_cache->stride[i]; p.os[i] = out->stride[i];
    }
    p.kv_lengths = kv_lengths;
    p.out = out->data;
    unsigned char *base = static_cast<unsigned char *>(scratch);
    p.counters = reinterpret_cast<int32_t *>(base);
    p.status = reinterpret_cast<int32_t *>(base + kStatusOff);
    p.partials = reinterpret_cast<float *>(base + kPartialsOff);
    rc = fd::launch_simt(p, (int)G, st);
    return rc == 0 ? FD_OK : (rc == -2 ? FD_ERR_UNSUPPORTED : FD_ERR_CUDA);
}
