// fd_launch.h -- kernel launchers called by the C ABI layer (fd_api.cu).
#pragma once

#include <cuda_runtime.h>

#include "fd_internal.h"

namespace fd {

// CUDA-core kernel (fd_simt.cu): every mode, head_dim 128 / 256.
int simt_tile_tokens();
int launch_simt(const Params &p, int num_ctas, cudaStream_t stream);

// Tensor-core kernel (fd_tc.cu, fd_tc_paged.cu): dense prefix (optionally
// causal) over flat or paged caches and index gather; bf16 caches at head_dim
// 128 / 256 with up to 64 packed rows, int8 at head_dim 128 / 256 with up to
// 32 (flat dense int8: more, in parts of a kv head's query heads, see
// tc_int8_row_parts); one block per SM.
int tc_tile_tokens();
// Work units the split charges per segment start (Params::seg_units).
int tc_seg_units(const Params &p);
bool tc_supports(const Params &p);
// Flat dense int8 caches with more than 32 rows (n_q x g): the fewest parts
// k, k dividing g, such that n_q * g / k <= 32 (the launch then serves g / k
// query heads per part and reads each kv head's caches k times); 0 if none.
int tc_int8_row_parts(int n_q, int g);
int launch_tc(const Params &p, int num_ctas, cudaStream_t stream);
// Paged caches (fd_tc_paged.cu); tc_supports covers them.
bool tc_supports_paged(const Params &p);
int launch_tc_paged(const Params &p, int num_ctas, cudaStream_t stream);
// Flat int8 caches, dense prefix and gather (fd_tc_int8.cu).
int launch_tc_int8(const Params &p, int num_ctas, cudaStream_t stream);
// Masked prefix over flat bf16 caches: each tile finds its visible chunks in
// place (fd_tc_masked.cu), or, with int32 scratch at p.mlist of
// tc_mask_list_ints(B, cap) entries, a pass lists the visible chunks and the
// decode walks only those (fd_tc_masked_list.cu).
int launch_tc_masked(const Params &p, int num_ctas, cudaStream_t stream);
int64_t tc_mask_list_ints(int64_t B, int64_t cap);
int launch_tc_masked_list(const Params &p, int num_ctas, cudaStream_t stream);
// Fused append over flat bf16 caches (fd_tc_append.cu): a cooperative launch,
// so num_ctas may not exceed the blocks resident at once (else -2).
int launch_tc_append(const Params &p, int num_ctas, cudaStream_t stream);

// Block top-k selection for the gather lists (fd_topk.cu): one thread block
// per (sequence, query row); n_blocks <= kTopkMaxBlocks (their keys live in
// shared memory).
constexpr int kTopkMaxBlocks = 32768;
int topk_max_blocks();
int launch_topk(const float *scores, int B, int n_q, int n_blocks, const int32_t *kv_lengths,
                int block_size, int top_k, int32_t *idx, cudaStream_t stream);

}  // namespace fd
