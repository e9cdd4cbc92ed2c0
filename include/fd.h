/*
 * fd.h -- C ABI of libfd.so: length-aware GQA decode attention over a
 * preallocated KV cache, for NVIDIA GB300 (sm_103a).
 *
 * What the calls compute.  For sequence b, query row i, query head h and
 * kv head hk = h / (Hq / Hkv):
 *
 *     out[b,i,h,:] = sum_{j in V} softmax_j(scale * q[b,i,h,:] . k[b,hk,j,:]) v[b,hk,j,:]
 *
 * over the visible cache positions V, and 0 where V is empty.
 *   - fd_decode / fd_decode_int8: V = the filled prefix 0 .. L-1 with
 *     L = kv_lengths[b] read on the device, so the call never touches the
 *     unused tail of the cache ("Qwen3.5 text generation attends over the
 *     full KV capacity", ComfyUI #16509: problem statement and the
 *     length-aware FixedKV path).  With causal != 0 the n_q query rows are
 *     the newest n_q positions of the cache (the decode token plus MTP
 *     drafts already written at L-n_q .. L-1) and row i sees 0 .. L-n_q+i
 *     (same issue, list item 2 and "Existing Solutions": a bottom-right
 *     aligned causal window, up to 6 rows).
 *     fd_decode_paged computes the same over a paged cache,
 *     fd_decode_append after writing the step's new rows into the cache, and
 *     fd_decode_masked with an additive mask over the prefix.
 *   - fd_decode_gather: V = the cells listed for that (b, i) in idx
 *     ("attend the selected cells instead of masking the window",
 *     llama.cpp #28244, Conversation; "gather-based sparse attention for
 *     QSA decode", llama.cpp #28213: per-token lists for multi-row verify);
 *     fd_decode_gather_bias adds a bias per list entry, and fd_topk_blocks
 *     builds the lists from block scores.
 * The prefix is split across thread blocks and the last block to finish a
 * (sequence, kv head) combines the splits inside the same launch
 * (comfy-kitchen #239, "GQA decode"); the query heads of one GQA group share
 * each K/V tile.
 *
 * Conventions shared by every call.
 *   - Tensors are described by fd_tensor: a data pointer, a dtype, 4 sizes
 *     and 4 strides counted in ELEMENTS.  The innermost (head_dim) stride
 *     must be 1.  Device pointers unless stated otherwise.
 *   - q      : [B, n_q, Hq, d] bf16.
 *   - caches : [B, Hkv, cap, d] bf16 (fd_decode, fd_decode_gather) or int8
 *              (fd_decode_int8); any strides that are multiples of 16 bytes,
 *              so the canonical [B, Hkv, cap, d] and the token-major
 *              [B, cap, Hkv, d] (seen through a transpose) both work; the
 *              data pointer must be 16-byte aligned.
 *   - out    : [B, n_q, Hq, d] bf16 or fp32 (round to nearest even for bf16).
 *   - d (head_dim) is 128 or 256; 1 <= n_q <= 6; Hq % Hkv == 0;
 *     (Hq / Hkv) * n_q <= 64 query rows share one kv head per launch unit.
 *   - The caller owns every tensor, kv_lengths and idx.  The library owns
 *     only the workspace (fd_workspace_create) and never allocates, frees or
 *     synchronises inside a decode call, and never reads device data on the
 *     host, so the calls can be captured in a CUDA graph and replayed with
 *     new lengths or index lists written on the device.
 *   - Work is queued on opts->stream (a cudaStream_t; NULL = the legacy
 *     default stream).  One workspace serves one stream at a time.
 *   - Return value: FD_OK, or a negative FD_ERR_* code.  Every argument is
 *     checked on the host before any CUDA call; on error nothing is
 *     launched.  FD_ERR_CUDA reports a launch failure (cudaGetLastError).
 *   - Bad device-side data (a length outside [0, cap], an index >= cap) never
 *     faults: the value is clamped or the cell skipped, and a sticky bit is
 *     set in the workspace status word (fd_get_device_status).
 */
#ifndef FD_H
#define FD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define FD_OK 0
#define FD_ERR_ARG (-1)          /* null pointer, bad shape/dtype/stride   */
#define FD_ERR_UNSUPPORTED (-2)  /* head_dim, n_q or group size not served */
#define FD_ERR_ALIGN (-3)        /* pointer or stride not 16-byte aligned  */
#define FD_ERR_WORKSPACE (-4)    /* missing or too small workspace         */
#define FD_ERR_CUDA (-5)         /* CUDA runtime error                     */
#define FD_ERR_SCRATCH (-6)      /* problem exceeds fd_decode_noalloc's fixed scratch */

/* dtypes */
#define FD_BF16 0
#define FD_F32 1
#define FD_I8 2
#define FD_I32 3

/* sticky device status bits (fd_get_device_status) */
#define FD_DEV_BAD_LENGTH 1      /* some kv_lengths[b] outside [0, cap]    */
#define FD_DEV_BAD_INDEX 2       /* some idx entry >= cap (skipped)        */
#define FD_DEV_INTERNAL 4        /* a bounded internal wait gave up; the
                                    call's output is not valid              */

/* kernel selection (fd_opts.kernel); AUTO takes the tensor-core kernel for
 * the calls it serves when q's base pointer and strides are 16-byte aligned
 * (q is read through a TMA tensor map there), the CUDA-core kernel
 * otherwise */
#define FD_KERNEL_AUTO 0
#define FD_KERNEL_SIMT 1         /* CUDA-core kernel, every mode           */
#define FD_KERNEL_TC 2           /* tensor-core (tcgen05) kernel: bf16
                                    caches (head_dim 128/256, up to 64
                                    rows) and int8 caches (head_dim
                                    128/256, up to 32 rows; flat dense
                                    int8 with more rows in parts, see
                                    fd_decode_int8), flat or paged
                                    (pools whose rows form one strided 2-D
                                    array), the fused append and the
                                    masked prefix over flat bf16 caches,
                                    and gather over bf16 or int8 caches
                                    whose rows form one strided 2-D array;
                                    16-byte aligned q (else
                                    FD_ERR_UNSUPPORTED)                    */

#define FD_MAX_ROWS 64           /* query rows per kv head per launch unit */

typedef struct fd_tensor {
    void *data;
    int32_t dtype;               /* FD_BF16, FD_F32, FD_I8, FD_I32          */
    int32_t ndim;                /* 1 .. 4                                  */
    int64_t shape[4];
    int64_t stride[4];           /* in elements                             */
} fd_tensor;

/* Opaque device workspace: per-split partial results, one completion counter
 * per (sequence, kv head) and the sticky status word. */
typedef struct fd_workspace fd_workspace;

typedef struct fd_opts {
    void *stream;                /* cudaStream_t, NULL = legacy default      */
    fd_workspace *ws;            /* required                                 */
    int32_t num_ctas;            /* 0 = auto (from the SM count); > 0 forces
                                    the number of thread blocks, which sets
                                    the split count                          */
    int32_t kernel;              /* FD_KERNEL_*                              */
    float scale;                 /* fd_decode_gather only: 0 = 1/sqrt(d)     */
    int32_t wait_limit_us;       /* tensor-core kernel: bound on each of its
                                    internal waits, in microseconds; 0 = the
                                    default of 2 s.  A wait that runs out sets
                                    FD_DEV_INTERNAL and the launch ends (its
                                    output is then not valid).  Tests of that
                                    path shorten it; 1 .. 2e6.              */
    int32_t reserved[2];         /* must be zero                             */
} fd_opts;

/*
 * Dense prefix decode (bf16 cache).
 *   q [B, n_q, Hq, d] bf16; k_cache, v_cache [B, Hkv, cap, d] bf16;
 *   kv_lengths: device int32[B], L_b = number of filled positions;
 *   n_q: query rows (must equal q->shape[1]); causal: 0 or 1;
 *   scale: multiplies q.k (usually 1/sqrt(d));
 *   out [B, n_q, Hq, d] bf16 or fp32.
 */
int fd_decode(const fd_tensor *q, const fd_tensor *k_cache,
              const fd_tensor *v_cache, const int32_t *kv_lengths,
              int32_t n_q, int32_t causal, float scale, const fd_tensor *out,
              const fd_opts *opts);

/*
 * Dense prefix decode over an int8 cache with one fp32 scale per
 * (sequence, kv head, position): k = k_code * k_scale[b, hk, j], likewise v
 * (comfy-kitchen #239, commit list: bounded paged INT8 decode cache; the
 * cache here is not paged).  k_scale, v_scale: fp32 [B, Hkv, cap] with any
 * strides.  Other arguments as fd_decode.
 * On the tensor-core kernel the products run on fp16 operands: the codes
 * convert exactly, q is rounded to fp16 (exact for bf16 values of magnitude
 * 2^-14 .. 65504; larger ones saturate at 65504), and each softmax weight
 * (at most 16 before normalisation) times the position's v scale is held
 * in fp16 with about 2^-22 relative error, saturating at 65504 (a v scale
 * above 4094, i.e. dequantised |v| above about 5.2e5, can saturate).  The
 * CUDA-core kernel has no such range limit.  The same holds for every
 * int8 call (paged and gather).
 * The tensor-core kernel takes up to 32 rows (n_q * g) at once.  With more,
 * it serves each kv head's query heads in k parts of g / k heads, k the
 * fewest dividing g that bring n_q * g / k to 32 or fewer, each part a
 * segment of its own that reads the kv head's prefix again (k times the
 * cache bytes); the workspace then needs B * Hkv * k segments (B * Hq always
 * suffices).  Under FD_KERNEL_AUTO a workspace without that room, or a
 * shape with no such k (g = 1), takes the CUDA-core kernel, which reads the
 * prefix once; FD_KERNEL_TC returns FD_ERR_WORKSPACE or FD_ERR_UNSUPPORTED.
 */
int fd_decode_int8(const fd_tensor *q, const fd_tensor *k_cache,
                   const fd_tensor *v_cache, const fd_tensor *k_scale,
                   const fd_tensor *v_scale, const int32_t *kv_lengths,
                   int32_t n_q, int32_t causal, float scale,
                   const fd_tensor *out, const fd_opts *opts);

/*
 * Index-gather decode (bf16 cache).
 *   idx: device int32 [B, n_q, idx_len], contiguous (may be NULL when idx_len
 *   is 0: every output row is then 0); one list per (sequence,
 *   query row), shared by all heads of that row.  Entries < 0 are padding;
 *   entries >= cap are skipped and flag FD_DEV_BAD_INDEX.  Lists are read as
 *   given: a cell listed twice counts twice (distinct cells reproduce the
 *   masked path exactly).  No length and no causal mask apply: the list is
 *   the visible set.  Scale: opts->scale, or 1/sqrt(d) when 0.
 *   On the tensor-core kernel with opts->num_ctas = 0, lists of 2 to 16
 *   tiles of 128 entries whose (sequence, query row, kv head) lists all fit
 *   the device at once run as thread-block clusters, one per list, whose
 *   blocks merge their partial results through distributed shared memory
 *   instead of the workspace (the list length alone decides).
 */
int fd_decode_gather(const fd_tensor *q, const fd_tensor *k_cache,
                     const fd_tensor *v_cache, const int32_t *idx,
                     int32_t idx_len, const fd_tensor *out,
                     const fd_opts *opts);

/*
 * Gather lists from block scores (no counterpart call in the pages; the
 * step they ask for next): for each (sequence b, query row i), top_k of the
 * blocks are selected by score and only the winners are expanded to cells
 * ("qwen4exp : gather-based sparse attention for QSA decode", llama.cpp
 * #28213, review discussion: take top-k over blocks and expand only the
 * winners, instead of selecting over every cell).
 *   scores: device fp32 [B, n_q, n_blocks], contiguous; block j covers cells
 *     j*block_size .. (j+1)*block_size - 1.  Scores must not be NaN.
 *   kv_lengths: device int32 [B]; L_b clamped to [0, n_blocks*block_size].
 *     The candidates of row (b, i) are the blocks whose first cell is below
 *     L_b; the top_k highest scores win, ties going to the lower index
 *     (-0 and +0 tie).
 *   idx: device int32 [B, n_q, top_k*block_size], contiguous, written: the
 *     winners in increasing block order, each as its block_size cells, cells
 *     at or past L_b as -1, padded with -1 when fewer than top_k blocks are
 *     candidates.  The result feeds fd_decode_gather (idx_len =
 *     top_k*block_size).
 *   n_blocks <= 32768 (FD_ERR_UNSUPPORTED beyond); n_blocks*block_size below
 *   2^31.  Queued on `stream`; allocates nothing, reads nothing back,
 *   graph-capturable.  Returns FD_OK or a negative FD_ERR_* code.
 */
int fd_topk_blocks(const float *scores, int32_t B, int32_t n_q,
                   int32_t n_blocks, const int32_t *kv_lengths,
                   int32_t block_size, int32_t top_k, int32_t *idx,
                   void *stream);
/*
 * Index-gather decode over an int8 cache with per-position fp32 scales: as
 * fd_decode_gather, with k = k_code * k_scale[b, hk, cell] and v likewise,
 * k_scale / v_scale as in fd_decode_int8.  The gather measurements of
 * "qwen4exp : gather-based sparse attention for QSA decode" (llama.cpp
 * #28213, Additional information and review discussion) all run over a q8_0
 * (8-bit) KV cache.  The tensor-core kernel serves head_dim 128 / 256 with up
 * to 32 query rows per list (fetching each listed cell's codes with
 * tile::gather4); the CUDA-core kernel serves the rest.
 */
int fd_decode_gather_int8(const fd_tensor *q, const fd_tensor *k_cache,
                          const fd_tensor *v_cache, const fd_tensor *k_scale,
                          const fd_tensor *v_scale, const int32_t *idx, int32_t idx_len,
                          const fd_tensor *out, const fd_opts *opts);
/*
 * Index-gather decode with a per-entry score bias: as fd_decode_gather, and
 * bias[b, i, t] (fp32, device, [B, n_q, idx_len] contiguous, aligned with
 * idx) is added to the scaled score of list entry t ("qwen4exp :
 * gather-based sparse attention for QSA decode", llama.cpp #28213, Overview:
 * the mask entries are gathered with the cells).  An entry whose bias is
 * -inf is dropped, exactly as if it were padding; every other bias must be
 * finite.  bias = NULL is fd_decode_gather.
 */
int fd_decode_gather_bias(const fd_tensor *q, const fd_tensor *k_cache,
                          const fd_tensor *v_cache, const int32_t *idx,
                          const float *bias, int32_t idx_len,
                          const fd_tensor *out, const fd_opts *opts);
/*
 * Dense prefix decode with an additive mask, skipping hidden chunks: as
 * fd_decode, and mask[b, i, j] (fp32, device, [B, n_q, cap], positions
 * contiguous) is added to the scaled score of query row i at position j;
 * -inf hides the position.  A 32-position chunk that the mask and the window
 * hide for every query row of a sequence is not read at all: the masked scan
 * whose cost follows the visible chunks ("qwen4exp : gather-based sparse
 * attention for QSA decode", llama.cpp #28213, Metal measurements: the
 * FA-vec kernel skips fully masked 32-cell chunks).  Mask values must be
 * finite or -inf.  Both kernels serve it: the CUDA-core kernel skips a
 * hidden chunk (its tiles are 32 positions); the tensor-core kernel, whose
 * tiles are 128 positions, loads each tile as four 32-position chunks and
 * copies only the chunks some query row sees.  When the workspace holds
 * fd_masked_list_bytes(B, cap) bytes past the call's split partials
 * ((B*Hkv + num_ctas) slots of slot_floats(rows, d) floats, rows = (Hq/Hkv)
 * * n_q, as fd_workspace_bytes counts them), a first pass on the stream lists
 * each sequence's visible chunks in that room and the tensor-core launch
 * walks only the listed chunks, four to a 128-position tile, so its time
 * follows the visible chunks, not the length; with less room each tile of the
 * prefix finds its visible chunks in place.  Positions the mask hides must
 * hold finite values (they lie in the filled prefix).  Other arguments as
 * fd_decode.
 */
int fd_decode_masked(const fd_tensor *q, const fd_tensor *k_cache,
                     const fd_tensor *v_cache, const int32_t *kv_lengths,
                     const fd_tensor *mask, int32_t n_q, int32_t causal,
                     float scale, const fd_tensor *out, const fd_opts *opts);
/*
 * Dense prefix decode with a fused K/V append (bf16 caches): one launch
 * writes the step's new rows into the caches and attends over the prefix
 * including them, as flash_attn_with_kvcache does with k / v and
 * cache_seqlens ("Qwen3.5 text generation attends over the full KV
 * capacity", ComfyUI #16509: Existing Solutions).  For sequence b with
 * base_b = kv_lengths[b] (clamped to [0, cap]):
 *   - k_new[b, i, hk, :] and v_new[b, i, hk, :] are written to cache
 *     positions base_b + i, i = 0 .. n_q - 1 (positions at or past cap are
 *     not written, and FD_DEV_BAD_LENGTH is set);
 *   - the result is fd_decode's with L_b = min(base_b + n_q, cap): the n_q
 *     query rows are the new tokens, and with causal != 0 row i sees
 *     positions 0 .. base_b + i;
 *   - with update_lengths = 1, kv_lengths[b] becomes L_b when the launch
 *     ends (0 leaves it unchanged).
 *   k_new, v_new: [B, n_q, Hkv, d] bf16, device, 16-byte aligned base and
 *   strides, inner stride 1 (the [B, n_q, Hkv, d] layout of q's new tokens).
 *   k_cache, v_cache and kv_lengths are written by the call (caller-owned).
 *   The tensor-core kernel runs it as a cooperative launch (every block
 *   resident; an explicit opts->num_ctas above that returns
 *   FD_ERR_UNSUPPORTED) and meets once at a grid-wide barrier after the
 *   writes; its launch counters live in the workspace, so calls sharing a
 *   workspace must not overlap.  Other arguments as fd_decode.
 */
int fd_decode_append(const fd_tensor *q, const fd_tensor *k_cache,
                     const fd_tensor *v_cache, const fd_tensor *k_new,
                     const fd_tensor *v_new, int32_t *kv_lengths,
                     int32_t update_lengths, int32_t causal, float scale,
                     const fd_tensor *out, const fd_opts *opts);
/*
 * Dense prefix decode over a paged cache: the same visible set, causal
 * window and result as fd_decode / fd_decode_int8, but cache position j of
 * sequence b lives in a pool of fixed-size pages, at row j % page_size of
 * page block_table[b * max_pages + j / page_size] (comfy-kitchen #239,
 * commit list and Description: a bounded paged int8 decode cache with
 * rollback).  Rolling a sequence back needs only a smaller kv_lengths[b];
 * pages past the length are never read.
 *   k_pages, v_pages: [num_pages, Hkv, page_size, d] bf16 or int8 (both the
 *     same), any strides that are multiples of 16 bytes, so the token-major
 *     pool [num_pages, page_size, Hkv, d] works through a transpose.
 *   k_scale, v_scale: NULL for bf16 pools; for int8 pools fp32
 *     [num_pages, Hkv, page_size] (any strides), one scale per cached row.
 *   block_table: device int32 [B, max_pages], contiguous, caller-owned.
 *     The logical capacity is cap = max_pages * page_size (below 2^31);
 *     kv_lengths[b] is clamped to [0, cap] (FD_DEV_BAD_LENGTH).  Only the
 *     entries of pages that hold positions < kv_lengths[b] are read; such an
 *     entry outside [0, num_pages) skips that page's positions and sets
 *     FD_DEV_BAD_INDEX.
 *   Other arguments as fd_decode.  The tensor-core kernel serves pools whose
 *   three outer strides are multiples of the smallest, itself at least d
 *   (every contiguous layout), with the row limits of the flat caches.
 */
int fd_decode_paged(const fd_tensor *q, const fd_tensor *k_pages,
                    const fd_tensor *v_pages, const fd_tensor *k_scale,
                    const fd_tensor *v_scale, const int32_t *block_table,
                    int32_t max_pages, const int32_t *kv_lengths, int32_t n_q,
                    int32_t causal, float scale, const fd_tensor *out,
                    const fd_opts *opts);
/*
 * Dense prefix decode that allocates nothing (no counterpart in the paper).
 *
 * For callers that cannot call cudaMalloc: an application whose own allocator
 * owns all device memory, a process under a hard device-memory cap, or a
 * plugin inside an engine that forbids allocation after start-up.  Computes
 * exactly what fd_decode computes (bf16 cache, optional causal window) on
 * `stream`, with the same arguments minus the workspace; num_ctas = 0 picks
 * the block count automatically.
 *
 * Its scratch (split partials, per-(sequence, kv head) completion counters
 * and an internal status word, which this call does not report) is a fixed
 * 8 MiB array in device memory that every GPU which loads libfd.so holds
 * until the process exits.  Limits: at most 4096
 * (sequence, kv head) pairs, and the split partials must fit: the block count
 * is lowered to fit, and a problem that cannot fit even with one block per
 * (sequence, kv head), or an explicit num_ctas that does not fit, returns
 * FD_ERR_SCRATCH before anything is launched.  Each call clears the counters
 * and status word on `stream` first (cudaMemsetAsync, which allocates
 * nothing).  All calls share the one array: calls that overlap on the GPU
 * race and must not be issued.  Every call whose stream is not being
 * captured looks up the array's device address (with the caller's device
 * current); a captured call reuses the address the last uncaptured call on
 * that device found.  So the first call on a device, and the first after a
 * device reset or in another context, must come before any stream capture
 * (a captured first call returns FD_ERR_CUDA).  Returns FD_OK or a negative
 * FD_ERR_* code.
 */
int fd_decode_noalloc(const fd_tensor *q, const fd_tensor *k_cache,
                      const fd_tensor *v_cache, const int32_t *kv_lengths,
                      int32_t n_q, int32_t causal, float scale,
                      const fd_tensor *out, void *stream, int32_t num_ctas);

/*
 * Workspace.  A launch unit ("segment") is one (sequence, kv head) in the
 * dense modes and one (sequence, query row, kv head) in gather mode; rows is
 * the number of query rows sharing it ((Hq/Hkv) * n_q dense, Hq/Hkv gather).
 * Size for the largest segment count, row count, head_dim and num_ctas any
 * call will use.  fd_workspace_create allocates device memory (cudaMalloc)
 * and zeroes the counters on `stream`; it is the only allocating call.
 * A workspace serves the calls of one stream at a time, in stream order: the
 * scratch of the split combine belongs to one stream-ordered launch at a
 * time, the rule comfy-kitchen #239 adopts for its GEMM workspace (commit
 * list: the workspace is tied to each launch in stream order).  Two streams
 * that may run decode calls at once need two workspaces.  Calls that do
 * overlap on one workspace can leave its counters inconsistent (results of
 * later calls are then wrong: a merge is skipped, or a masked call keeps an
 * older chunk list) until fd_workspace_reset.
 */
size_t fd_workspace_bytes(int64_t max_segments, int32_t max_rows,
                          int32_t head_dim, int32_t max_ctas);
int fd_workspace_create(int64_t max_segments, int32_t max_rows,
                        int32_t head_dim, int32_t max_ctas, void *stream,
                        fd_workspace **ws);
/* Clears the completion counters and the status word on `stream` (needed
 * only after a launch was aborted part-way; every completed launch leaves the
 * counters at zero). */
int fd_workspace_reset(fd_workspace *ws, void *stream);
/* Test hook for the failure path: sets every per-segment completion counter
 * to `value` on `stream`.  A negative value stands for counters an aborted
 * launch left behind: the next call whose blocks share the merge of a split
 * segment (the tensor-core kernel's cooperative launches over few segments)
 * then waits for pieces that never arrive, gives up after opts->wait_limit_us
 * and sets FD_DEV_INTERNAL, recording the wait in fd_get_device_diagnostics;
 * fd_workspace_reset restores the zeros.  Never needed in normal use. */
int fd_workspace_fill_counters(fd_workspace *ws, int32_t value, void *stream);
int fd_workspace_destroy(fd_workspace *ws);
/* Synchronously reads the sticky status word (FD_DEV_* bits). */
int fd_get_device_status(fd_workspace *ws, int32_t *status);
/* Synchronously reads 13 words: the status word; then, if FD_DEV_INTERNAL was
 * set by the tensor-core kernel, the id, tile counter and piece index of the
 * first internal wait that gave up; then the same three for the first wait
 * that gave up in each role (TMA producer, MMA issuer, softmax).  Zero where
 * nothing gave up.  Cleared by fd_workspace_reset. */
int fd_get_device_diagnostics(fd_workspace *ws, int32_t *words);

/* Number of thread blocks an auto launch of a dense call with this cache
 * dtype would use on the current device (host query; 0 on error).  max_units
 * bounds the launch's work units (tiles for the capacity plus fd_seg_units
 * per segment); 0 for no bound. */
int32_t fd_auto_num_ctas(int32_t kernel, int32_t head_dim, int32_t kv_dtype,
                         int32_t rows, int64_t max_units);
/* Cache positions per K/V tile for a kernel / head_dim / cache dtype. */
int32_t fd_tile_tokens(int32_t kernel, int32_t head_dim, int32_t kv_dtype);
/* Workspace bytes the tensor-core kernel's chunk list of a masked call over
 * B sequences of capacity cap takes past the call's split partials (the
 * list, the counts and the listing pass's staging area); 0 for B or cap
 * outside [1, 65535] or [1, 2^23], where no list is made. */
size_t fd_masked_list_bytes(int64_t B, int64_t cap);

/*
 * Host mirror of the device split partitioner, for inspection and tests.
 * The split is over work units: each non-empty segment holds seg_units units
 * (the fixed cost of a piece boundary, mapped to no tile) followed by one
 * unit per tile; num_ctas blocks take balanced consecutive unit ranges.
 * For segment lengths seg_len[0..nseg) (positions), tile size, num_ctas and
 * seg_units, writes for every segment the first thread block that works on
 * its tiles and the number of blocks that share them (0 for an empty
 * segment).  Returns the total unit count, or a negative FD_ERR_* code.
 */
int64_t fd_plan(const int64_t *seg_len, int64_t nseg, int32_t tile_tokens,
                int32_t num_ctas, int32_t seg_units, int32_t *first_cta,
                int32_t *n_pieces);
/* seg_units a launch of this kernel, head_dim and cache dtype uses (0 for
 * the CUDA-core kernel; AUTO is not resolved here). */
int32_t fd_seg_units(int32_t kernel, int32_t head_dim, int32_t kv_dtype);

const char *fd_status_string(int status);
int32_t fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_H */
