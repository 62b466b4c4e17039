// sv_internal.h -- launchers shared between the C-ABI translation unit and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

// One logits tensor [B][rows][V] (strides in elements) of element type dtype (0 fp32, 1 bf16).
struct Logits {
    const void *ptr;
    int64_t batch_stride;
    int64_t row_stride;
};

// Sampling path -----------------------------------------------------------------------
// Row statistics of B sequences of R = rows_a + rows_b rows: local rows [0, rows_a) come
// from `a`, [rows_a, R) from `b` (row rows_a + i of b is row i of tensor b).  One partial
// (M, S) per (row, 4 KB tile) is written to partial[(seq * R + row) * ntile + tile].
cudaError_t launch_stats_tiles(int dtype, bool vec, Logits a, int rows_a, Logits b, int R, int B, int V,
                               int ntile, float c, void *partial, cudaStream_t s);
// Merge the tile partials of every row, run the accept scan, write accepted_len, the
// accepted drafts and the -1 padding, and the per-sequence plan (k, mode).
cudaError_t launch_decide(int dtype, Logits t, Logits d, int B, int gamma, int V, int ntile,
                          float c, const int32_t *x, uint64_t seed, uint64_t offset,
                          const void *partial, void *rowstat, void *plan, int32_t *accepted_len,
                          int32_t *out_tokens, cudaStream_t s);
// Residual mass sum_j (p_j - q_j)+ of every residual tile of the stop row (sequences that
// rejected): csum[seq * nrt + tile].
cudaError_t launch_residual_tiles(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V,
                                  int nrt, float c, const void *rowstat, const void *plan, float *csum,
                                  cudaStream_t s);
// Inverse-CDF draw of the final token on the stop row of every valid sequence.
cudaError_t launch_draw(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V, int ntile, int nrt,
                        float c, uint64_t seed, uint64_t offset, const void *partial, const void *rowstat,
                        const void *plan, const float *csum, int32_t *out_tokens, cudaStream_t s);
// Test hook: (m, lse) per row from the partials.
cudaError_t launch_rowstats_finalize(int rows, int ntile, float c, float inv_t, const void *partial,
                                     float *m_out, float *lse_out, cudaStream_t s);
cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                            float *out, cudaStream_t s);

// Greedy / tree path ------------------------------------------------------------------
// The NaN-propagating maximum of every (row, 4 KB tile) of [B][R][V]: partial[row * ntile + tile].
cudaError_t launch_max_tiles(int dtype, bool vec, Logits t, int R, int B, int V, int ntile, void *partial,
                             cudaStream_t s);
// Row argmax from the tile maxima (the first position of the maximum, searched in the
// lowest tile that holds it), then the accept rule; both read t again for that one tile.
cudaError_t launch_greedy_finalize(int dtype, bool vec, Logits t, int B, int gamma, int V, int ntile,
                                   const void *partial, const int32_t *x, int32_t *accepted_len,
                                   int32_t *out_tokens, cudaStream_t s);
cudaError_t launch_tree_finalize(int dtype, bool vec, Logits t, int B, int N, int V, int ntile,
                                 const void *partial, const int32_t *parent, const int32_t *node_tokens,
                                 int max_depth, int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                                 cudaStream_t s);

}  // namespace sv
