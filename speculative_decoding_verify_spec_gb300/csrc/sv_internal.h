// sv_internal.h -- launchers shared between the C-ABI translation unit and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// One logits tensor [B][rows][V] (strides in elements) of element type dtype (0 fp32, 1 bf16).
struct Logits {
    const void *ptr;
    int64_t batch_stride;
    int64_t row_stride;
};

// Row r of sequence b as bytes (element size `bytes`).
__host__ __device__ inline const char *row_ptr(const Logits &L, int bytes, int64_t b, int64_t r) {
    return static_cast<const char *>(L.ptr) + (b * L.batch_stride + r * L.row_stride) * bytes;
}

// The sampling rules that share the draw and the re-draw: the chain (residual (p - q)+ after a
// rejection), a one-hot draft distribution (p without the rejected token), typical
// acceptance (the token at the stop drawn from p itself).
constexpr int kRuleSample = 0, kRuleOnehot = 1, kRuleTypical = 2;

// Extended-precision re-draw of near-boundary sampling sequences -----------------------
// decide marks a sequence whose accept test had |u q - p| < kRefineAcceptWindow * max(p, u q)
// (flag kRefineAccept); draw marks one whose threshold u'R lies within
// kRefineCdfWindow * R of a CDF boundary or that needed a rounding fallback (kRefineDraw),
// and lists every marked sequence: those with kRefineAccept on the rescan list (entries B ..
// 2B - 1 of the records), the others on the main list (entries 0 .. B - 1); refine redoes
// all of them in double-float arithmetic.  Control block (int32, zeroed by decide every
// call), followed by the per-sequence marks rflag[B]:
constexpr int kRefineCount = 0;     // sequences marked by this call
constexpr int kRefineMain = 1;      // entries on the main list
constexpr int kRefineAll = 2;       // entries on the rescan list
constexpr int kRefineStatus = 3;    // SV_ERR_TIMEOUT if a bounded wait of the re-draw gave up
constexpr int kRefineRedone = 4;    // sequences whose final token the re-draw wrote
constexpr int kRefineCtlWords = 8;
constexpr int kRefineDraw = 1, kRefineAccept = 2;
constexpr float kRefineAcceptWindow = 1e-6f;
// Draw prefixes are double-float, so the gap is limited by the unit masses' own fp32 error:
// a bonus draw's units are row-statistics tiles rescaled by one exponential each (~1e-7 of a
// tile's mass, the same for every logit of it), a residual draw's are direct sums.
constexpr float kRefineCdfWindow = 2e-7f;      // bonus draw from p (mode 0)
constexpr float kRefineCdfWindowRes = 6e-8f;   // residual draw (mode 1)
// Every draw window also holds kTokenWindow x min(1, S - 1) / S for each row the weights
// come from (S = sum 2^y, y = (x - M) c <= 0): one fp32 weight 2^y is off by at most ~2.5e-7
// (ex2.approx's own error, measured at 1.42e-7 relative over [-40, 0], plus the argument's
// rounding, 2^y |y| <= 0.53, and the product with 1 / S), except the row maximum's,
// 2^0 = 1 exactly; so one other token of weight up to min(1, S - 1) can move a boundary by
// that much -- on a row carried by a few tokens more than the windows above, which are set
// by the many small, independent errors of spread-out rows.
constexpr float kTokenWindow = 3e-7f;
__host__ __device__ inline float token_window(float S) { return kTokenWindow * fminf(1.f, S - 1.f) / S; }
// What draw records about a listed sequence (the re-draw's first read).
struct RefineInfo {
    int seq, flag, k, mode;  // plan (k, mode) as decided in fp32
    float Mt, St, Md, Sd;    // fp32 (max, sum) of target / draft row k (Md, Sd unused for a bonus draw)
};
// Re-draw scratch (units of 64 logits, refine_units(V) of them per row): per main-list
// sequence 5 rows of double-float unit sums and one of near-logit counts; the rescan list
// is taken kRescanChunk sequences at a time, (2 gamma + 1) rows of unit sums each.
constexpr int kRescanChunk = 16;
inline int64_t refine_units(int V) { return (int64_t(V) + 63) / 64; }

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
                          int32_t *out_tokens, int *rflag, int *rctl, int *rbar, cudaStream_t s);
// Residual mass sum_j (p_j - q_j)+ of every residual tile of the stop row (sequences that
// rejected): csum[seq * nrt + tile].
cudaError_t launch_residual_tiles(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V,
                                  int nrt, float c, const void *rowstat, const void *plan, float *csum,
                                  cudaStream_t s);
// One sequence whose 2 gamma + 1 rows hold at most kSingleTiles tiles: the whole sampling
// call (the four kernels' stages and the re-draw) in one kernel of one CTA; same workspace.
constexpr int kSingleTiles = 256;
bool single_sample_fits(int B, int gamma, int ntile);
cudaError_t launch_single_sample(int dtype, bool vec, Logits t, Logits d, int gamma, int V, int ntile, int nrt,
                                 float c, float T, uint64_t seed, uint64_t offset, const int32_t *x, void *partial,
                                 void *rowstat, void *plan, float *csum, int32_t *accepted_len, int32_t *out_tokens,
                                 int *rctl, int *rbar, RefineInfo *rinfo, void *rsum, int *ramb, void *rresc,
                                 cudaStream_t s);
// Inverse-CDF draw of the final token on the stop row of every valid sequence, then the
// extended-precision re-draw of every sequence it or decide marked (one cooperative grid;
// rbar: its grid barrier's words; rsum, ramb, rresc: the re-draw's scratch, see above).
// rule: kRuleSample / kRuleOnehot / kRuleTypical (which rows the rescan reads, and its test);
// R: rows per sequence in partial / rowstat; lavail: rows a lazy walk read per sequence
// (NULL: all of them).
cudaError_t launch_draw_refine(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V, int ntile, int nrt,
                               float c, float T, uint64_t seed, uint64_t offset, int rule, int R, const int *lavail,
                               const int32_t *x, const void *partial,
                               const void *rowstat, const void *plan, const float *csum, int32_t *accepted_len,
                               int32_t *out_tokens, int *rctl, int *rbar, RefineInfo *rinfo, void *rsum, int *ramb,
                               void *rresc, bool early, cudaStream_t s);
// Extended-precision re-walk of near-boundary tree-sampling sequences -----------------
// The walk marks sequence b (mark[b] = 1, else 0, every call) when one of its fp32
// decisions came near enough to flipping: an accept test with |u q - p| below
// kTreeAcceptWindow x (max(p, u q) + the size of p's terms), a residual mass below
// kTreeMassWindow x (1 + A), less than kTreeQMassWindow of q's mass left, more removed
// tokens than it tracks, or a final draw whose threshold lies within kTreeCdfWindow x
// (total + A) of a CDF boundary (A: the walk's coefficient; total: the draw's mass; the
// draw's prefixes are fp64 sums of the fp32 weights, so the gap is that of the weights'
// own rounding, measured below 7e-9 (total + A) on the workloads).  It records
// the first kTreeRecNodes nodes it reached (rec: node, M_t, M_d, has children; rlen: how
// many).  The re-walk redoes every marked sequence in double-float arithmetic:
// kMaxTreeRefine clusters, the first kMaxTreeRefine marked sequences with exponentials the
// whole grid precomputed (slots), later ones computing them in their cluster.  Control block (int32, zeroed by the walk; words other than these stay 0):
// Mark bits of a tree walk: a decision on the path came near flipping (the re-walk starts
// at the root), or only the final draw at the reached node did (the path is certain: the
// re-walk starts at that node).
constexpr int kTrMarkPath = 1, kTrMarkFinal = 2;
constexpr int kTrMarked = 0;  // sequences the last call marked
constexpr int kTrRedone = 4;  // sequences redone (every marked one)
constexpr int kTrFinalDone = 5;  // slots (bit j) whose final draw the exponentials kernel redid
constexpr int kTrCtlWords = 8;  // (words 1, 2 and 3: that kernel's grid barrier; 3 is the status)
constexpr int kMaxTreeRefine = 8;
constexpr int kTreeRecNodes = 8;
constexpr float kTreeAcceptWindow = 1e-6f;
constexpr float kTreeMassWindow = 1e-6f;
constexpr float kTreeQMassWindow = 1e-5f;
constexpr float kTreeCdfWindow = 4e-8f;
constexpr int kTreeRefineCluster = 16;  // at most this many CTAs of the re-walk's cluster per sequence
struct df;
// Workspace of the re-walk, K = min(max_depth + 1, kTreeRecNodes) positions, nunit =
// tree_refine_units(V):  ctl [kTrCtlWords]; mark, rlen [B]; rec [B][K] float4;
// et [kMaxTreeRefine][K][2][V] and us [kMaxTreeRefine][K][2][nunit] double-float (the
// exponentials of the recorded rows and their unit sums); npos [kMaxTreeRefine][K] int;
// um [2][kMaxTreeRefine][nunit] (two buffers: passes in turn), part [kMaxTreeRefine][2][cluster][2] double-float; pmax
// [kMaxTreeRefine][cluster][2] float; pcnt [kMaxTreeRefine][cluster] int.
struct TreeRefineWs {
    int *ctl, *mark, *rlen;
    float4 *rec;
    df *et, *us;
    int *npos;
    df *um, *part;
    float *pmax;
    int *pcnt;
};
constexpr int kTreeRefineUnit = 256;  // logits per unit of the re-walk's passes (one warp)
__host__ __device__ inline int tree_refine_units(int V) {
    return int((int64_t(V) + kTreeRefineUnit - 1) / kTreeRefineUnit);
}
inline int tree_rec_nodes(int max_depth) { return max_depth + 1 < kTreeRecNodes ? max_depth + 1 : kTreeRecNodes; }
inline size_t tree_refine_smem(int N, int max_depth) { return size_t(13 * N + max_depth + 1) * 4; }
// The exponentials of the listed sequences' recorded rows (every resident CTA; for a
// sequence marked only at its final draw, the reached node's rows alone) and the final
// re-draw of those marked only there (the same grid), then the re-walk of the rest (one
// cluster of 16 CTAs per listed sequence where the device holds one, else 8).
// accepted_len: the walk's outputs (the depth it reached).
cudaError_t launch_tree_exp(int dtype, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                            const int32_t *node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                            int without_replacement, int K, TreeRefineWs ws, int32_t *accepted_len,
                            int32_t *out_tokens, int32_t *out_path, cudaStream_t s);
cudaError_t launch_tree_rewalk(int dtype, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                               const int32_t *node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                               int without_replacement, int K, TreeRefineWs ws, int32_t *accepted_len,
                               int32_t *out_tokens, int32_t *out_path, cudaStream_t s);
// Token-tree sampling (multi-round rejection), a cluster of CTAs per sequence reading the
// rows of the nodes its walk reaches.  c = log2(e) / T; umass: [B][nunit] floats of
// scratch, nunit = ceil(V / res_tile_elems); cstat: [B][kTreeSampleCluster][2] float2;
// rw, K: the re-walk's control block, marks and records (below).
constexpr int kTreeSampleCluster = 4;  // at most this many CTAs (SMs) per sequence of the walk
cudaError_t launch_tree_sample(int dtype, bool vec, Logits t, Logits d, int B, int N, int V,
                               const int32_t *parent, const int32_t *node_tokens, int max_depth, float c, uint64_t seed,
                               uint64_t offset, int without_replacement, int nunit, float *umass, float2 *cstat,
                               TreeRefineWs rw, int K, int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                               cudaStream_t s);
// Lazy greedy verification, one CTA per sequence reading only the rows of accepted nodes:
// a tree (parent[N], tokens [B][N]) or, with chain, the chain of draft tokens [B][N - 1].
cudaError_t launch_greedy_walk(int dtype, bool vec, Logits t, int B, int N, int V, bool chain, const int32_t *parent,
                               const int32_t *tokens, int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                               int32_t *out_path, cudaStream_t s);
// Prompt-lookup drafting: history [B][stride] with lengths[B]; drafts [B][k], count [B].
constexpr int kMaxNgram = 64;
cudaError_t launch_ngram_draft(const int32_t *history, int64_t stride, const int32_t *lengths, int B, int n, int k,
                               int pad, int32_t *drafts, int32_t *count, cudaStream_t s);
// Test hook: one CTA through the re-draw's grid barrier expecting `expected` arrivals.
cudaError_t launch_wait_selftest(int *ctl, int expected, uint64_t limit_ns, cudaStream_t s);
// Test hook: exp(hi + lo) in double-float for n arguments <= 0.
cudaError_t launch_exp_df(const float *y_hi, const float *y_lo, int n, float *out_hi, float *out_lo,
                          cudaStream_t s);
// Test hook: (m, lse) per row from the partials.
cudaError_t launch_rowstats_finalize(int rows, int ntile, float c, float inv_t, const void *partial,
                                     float *m_out, float *lse_out, cudaStream_t s);
cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                            float *out, cudaStream_t s);

// Level-synchronous lazy walks (sv_level.cu) --------------------------------------------
struct LevelArgs {
    Logits t, d;                     // d: draft rows (the sampling chain only)
    int B, gamma, V, ntile;
    int R;                           // rows per sequence in partial / rowstat: 2 gamma + 1 (chain), else gamma + 1
    float c;                         // log2(e) / T
    const int32_t *x;                // draft tokens [B][gamma]
    uint64_t seed, offset;
    float epsilon, delta;            // typical acceptance's threshold
    float2 *partial;                 // [B][R][ntile] (M, S) per 4 KB tile
    float *zpart;                    // [B][R][ntile] Z per tile (typical acceptance)
    float *xval;                     // [B][R] the logit at the draft token of each row read
    float2 *rowstat;                 // [B][R] (M, S) of every row read
    int2 *plan;                      // [B] (stop row, kind of draw: 0 from p, 1 residual, 2 p without x_k)
    int32_t *accepted_len, *out_tokens;
    int *rctl, *rbar;                // the draw kernel's re-draw control words and barrier (zeroed here)
    int *lctl;                       // [8] this kernel's grid barrier, then [gamma + 2] level list lengths
    int *lact;                       // [2][B] the sequences of the current and the next level
    int *tcnt;                       // [B] tiles of the current step counted in
    int *lstate;                     // [B] bit 0 walking, bit 1 marked for the rescan
    int *lavail;                     // [B] rows 0 .. lavail - 1 read (what the rescan may use)
};
// The walk (a cooperative grid, one CTA of 768 threads per SM), after zeroing lctl's
// barrier words and list lengths and tcnt.  A step fetches one level's rows, or every
// remaining level's once that is at most 64 MB, and the finishing warp walks them in order.
cudaError_t launch_level(int rule, int dtype, bool vec, const LevelArgs &a, cudaStream_t s);

// Host-side helpers shared by the entry points ----------------------------------------
inline int elem_bytes(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }
// Logits per 4 KB tile of the streaming kernels (32 lanes x 8 sixteen-byte vectors).
inline int tile_elems_of(sv_dtype d) { return 32 * 8 * (16 / elem_bytes(d)); }
inline int ntile_of(int V, sv_dtype d) { return int((int64_t(V) + tile_elems_of(d) - 1) / tile_elems_of(d)); }
// 16-byte vector loads are legal when the base and both strides keep every row aligned.
inline bool vec_ok(const void *p, int64_t sb, int64_t sr, sv_dtype d) {
    const int64_t e = elem_bytes(d);
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((sb * e) % 16 == 0) && ((sr * e) % 16 == 0);
}
// Records stage event s of the calling thread's list (spec_verify_set_stage_events), if any;
// stage 0 is "before the first kernel".
cudaError_t mark_stage(int s, cudaStream_t stream);

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
