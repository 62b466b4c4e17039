/*
 * spec_verify.h -- C ABI of libspecverify, the speculative-decoding verification step on
 * one GPU (hand-written sm_103a CUDA kernels).
 *
 * Sources (page title -- section):
 *   [SD] "7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead": "The rule"
 *        (accept x with probability min(1, p(x)/q(x)), else resample from the normalised
 *        residual (p - q)+), "Extending to a chain of gamma draft tokens" (left to right,
 *        stop at the first rejection, bonus token from row gamma when all are accepted;
 *        temperature 0 = longest matching prefix), "A From-Scratch Implementation"
 *        (apply_temperature on BOTH models; row i of the target predicts the token after
 *        draft i), "Tree Attention" and Exercise 5 (verify_tree_greedy on a parent-indexed
 *        tree whose row i predicts the token after node i).
 *   [MS] "Medusa, EAGLE and self-speculation": speculative_greedy (the correction token is
 *        the argmax at the first mismatching row).
 *   [HB] "Speculative Decoding: Draft Models, EAGLE, and How to Actually Use It": "The
 *        Algorithm" (steps 1-4).
 *
 * Conventions shared by every entry point
 *   - Every array argument is a DEVICE pointer; the caller owns all memory.  The library
 *     allocates nothing and keeps no state between calls, apart from the optional,
 *     thread-local timing events of spec_verify_set_stage_events and the fixed scratch
 *     array of spec_verify_greedy_noalloc.
 *   - Logits are [B][rows][V] with a contiguous last axis.  Strides are in ELEMENTS and may
 *     be 0 (broadcast).  Rows are read with 16-byte vector loads when the base pointer and
 *     both strides (times the element size) are multiples of 16 bytes, else element-wise.
 *   - Integer arrays (tokens, lengths, parents, paths) are int32, contiguous, row-major.
 *   - A call validates its arguments on the host and returns an error code BEFORE any
 *     work is enqueued; otherwise it enqueues its kernels on `stream` (a cudaStream_t;
 *     NULL = the legacy default stream) and returns without synchronising.  A launch
 *     failure returns SV_ERR_CUDA.
 *   - Bad data inside one sequence (a NaN, or for sampling a +inf or an all -inf row; a
 *     token outside [0, V)) is reported per sequence: accepted_len[b] = -1 and every output
 *     token of that sequence = -1.  Other sequences are unaffected.
 *   - `workspace` is caller-provided device scratch of at least
 *     spec_verify_workspace_size(...) bytes, 16-byte aligned.  Its contents need no
 *     initialisation.  After the call only the status words that spec_verify_status_offset
 *     locates mean anything.  Calls that run concurrently need distinct workspaces.
 *   - The sampling entries decide in fp32 and redo EVERY sequence whose fp32 decision came
 *     near enough to its boundary to be in doubt in double-float arithmetic (~48 bits), so
 *     their result is the exact rule's except where a comparison's exact margin is below
 *     ~1e-12 relative.  Their device-side outcome (sequences marked, sequences redone, and a
 *     status that is SV_OK unless a bounded device wait gave up) is in the workspace at
 *     spec_verify_status_offset once the stream has completed.
 *   - A round emits accepted_len[b] + 1 tokens (always >= 1) [SD "Extending to a chain"].
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* a size, stride, pointer or temperature is out of range */
    SV_ERR_UNSUPPORTED = 2, /* dtype or mode not supported */
    SV_ERR_CUDA = 3,        /* a CUDA launch failed; see cudaGetLastError semantics */
    SV_ERR_TIMEOUT = 4,     /* a bounded device wait gave up (re-draw status words) */
    SV_ERR_WORKSPACE = 5,   /* workspace NULL, too small or not 16-byte aligned */
    SV_ERR_CHECK = 6        /* bounds-checked build only: an internal index left its extent */
} sv_status;

typedef enum { SV_FP32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum {
    SV_MODE_SAMPLE = 0,    /* spec_verify_sample:      rows = gamma */
    SV_MODE_GREEDY = 1,    /* spec_verify_greedy:      rows = gamma */
    SV_MODE_TREE = 2,      /* spec_verify_tree_greedy: rows = N     */
    SV_MODE_ROW_STATS = 3, /* spec_verify_row_stats:   rows = rows_per_seq */
    SV_MODE_TREE_SAMPLE = 4, /* spec_verify_tree_sample: rows = N   */
    SV_MODE_SAMPLE_LAZY = 5, /* spec_verify_sample_lazy: rows = gamma */
    SV_MODE_TYPICAL = 6,     /* spec_verify_typical:     rows = gamma */
    SV_MODE_SAMPLE_ONEHOT = 7 /* spec_verify_sample_onehot: rows = gamma */
} sv_mode;

/* Limits checked on the host (SV_ERR_INVALID_ARG beyond them). */
#define SV_MAX_GAMMA 1024
#define SV_MAX_TREE_NODES 1024
#define SV_MAX_VOCAB (1 << 30)

/* Bytes of device workspace the given call needs (0 when B == 0).  Pure host function. */
size_t spec_verify_workspace_size(sv_mode mode, int B, int rows, int V, sv_dtype dtype);

/*
 * Sampling verification [SD "The rule", "Extending to a chain"; HB "The Algorithm"].
 *
 *   target_logits  [B][gamma+1][V]  row i predicts the token after draft i; row gamma is the
 *                                   bonus row.  Strides t_batch_stride, t_row_stride.
 *   draft_logits   [B][gamma][V]    the drafter's logits at the drafted positions (may be
 *                                   NULL when gamma == 0).  Strides d_batch_stride, d_row_stride.
 *   dtype          both logits arrays have this element type (fp32 or bf16).
 *   draft_tokens   [B][gamma]       x_0 .. x_{gamma-1}, drawn by the drafter from q.
 *   temperature    > 0 and finite; p = softmax(target / T), q = softmax(draft / T) (the
 *                  temperature applies to BOTH models).
 *   seed, offset   key the Philox4x32-10 uniforms: u(b, i, purpose) is word 0 of Philox
 *                  at counter (4 i + purpose, b, offset lo32, offset hi32) with key
 *                  (seed lo32, seed hi32), mapped to (w >> 8) * 2^-24.  purpose 0: the
 *                  accept test of draft i; purpose 1: the final draw on row i.  Callers vary
 *                  seed or offset between rounds.
 * Per sequence b: draft i is accepted iff u(b,i,0) * q_i(x_i) < p_i(x_i) (the strict test
 * u < min(1, p/q) with the division cleared).  The first rejection at k ends the round and
 * the token at k is drawn from (p_k - q_k)+ (if that residual is exactly 0, from p_k);
 * if all gamma are accepted, k = gamma and the bonus token is drawn from p_gamma.  A draw
 * is the inverse CDF in vocabulary order: the first j with r_0 + ... + r_j > u(b,k,1) * R.
 * Outputs:
 *   accepted_len   [B]           k, or -1 for bad data.
 *   out_tokens     [B][gamma+1]  x_0 .. x_{k-1}, the drawn token at k, then -1.
 */
sv_status spec_verify_sample(const void *target_logits, int64_t t_batch_stride,
                             int64_t t_row_stride, const void *draft_logits,
                             int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype, int B,
                             int gamma, int V, const int32_t *draft_tokens, float temperature,
                             uint64_t seed, uint64_t offset, int32_t *accepted_len,
                             int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Greedy verification [SD "Extending to a chain" (temperature 0); MS speculative_greedy].
 *
 *   target_logits  [B][gamma+1][V], draft_tokens [B][gamma].
 * a_i = argmax of row i (ties to the lowest index, values compared exactly after widening
 * to fp32).  n = the longest prefix with draft_tokens[b][i] == a_i.  Outputs:
 *   accepted_len [B] = n (or -1: a NaN in any row, or a draft token outside [0, V));
 *   out_tokens [B][gamma+1] = x_0 .. x_{n-1}, a_n, then -1.
 */
sv_status spec_verify_greedy(const void *target_logits, int64_t t_batch_stride,
                             int64_t t_row_stride, sv_dtype dtype, int B, int gamma, int V,
                             const int32_t *draft_tokens, int32_t *accepted_len,
                             int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Greedy token-tree verification [SD "Tree Attention", Exercise 5].
 *
 *   target_logits  [B][N][V]  row v predicts the token that follows node v.
 *   parent         [N]        parent[0] = -1, 0 <= parent[v] < v (parents before children);
 *                             one tree shared by the whole batch.
 *   node_tokens    [B][N]     the drafted token at node v ([b][0], the committed root, is
 *                             ignored).
 *   max_depth      >= the tree's depth; the width of the outputs is max_depth + 1.
 * Node v != 0 is accepted when node_tokens[b][v] == argmax(row parent[v]) and its parent is
 * accepted (the root always is).  v* = the deepest accepted node, the lowest index among
 * equally deep ones.  Outputs (each row max_depth+1 wide, -1 padded):
 *   accepted_len [B] = depth(v*);  out_tokens[b] = tokens on the path root -> v* without
 *   the root, then argmax(row v*) (the bonus);  out_path[b] = node ids root .. v* (out_path
 *   may be NULL).  A malformed tree, or one deeper than max_depth, makes every sequence -1;
 *   a NaN in any row of b, or a token of b outside [0, V), makes sequence b -1.
 */
sv_status spec_verify_tree_greedy(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, sv_dtype dtype, int B, int N, int V,
                                  const int32_t *parent, const int32_t *node_tokens,
                                  int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                                  int32_t *out_path, void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Token-tree SAMPLING verification by multi-round (recursive) rejection [SD "Tree
 * Attention", the paragraph on SpecInfer's rule].
 *
 *   target_logits  [B][N][V]  row v: the target's logits after the path to node v (p_v).
 *   draft_logits   [B][N][V]  row v: the drafter's logits at node v (q_v), from which v's
 *                             children were drawn; rows of leaves are never read.
 *   parent, node_tokens, max_depth: as spec_verify_tree_greedy.  Children are tested in
 *                             increasing node index (the order they were drawn).
 *   temperature, seed, offset: as spec_verify_sample (applied to both models).
 *   without_replacement       nonzero if each node's children were drawn from q_v without
 *                             replacement (q is then renormalised over the untested ones).
 * From the root: test the children of the current node in order with the single-candidate
 * rule (accept child c iff u q(x) < p(x), u = U(b, c - 1, purpose 0)); an accepted child
 * becomes the current node; a rejection replaces p by (p - q)+ normalised (and removes x
 * from q without replacement).  When all children are rejected the final token is drawn
 * from the last residual, at a leaf from p_v (inverse CDF, u' = U(b, v, purpose 1)).  A
 * chain-shaped tree gives spec_verify_sample's rule.  Outputs as spec_verify_tree_greedy:
 * accepted_len = depth of the final node, out_tokens = path tokens then the final token,
 * out_path = node ids (may be NULL).  Rows are read lazily, one cluster of 1, 2 or 4 CTAs
 * per sequence: only the rows of the nodes the walk reaches.  A malformed or too deep tree makes every sequence
 * -1; a token of b outside [0, V), or a row the walk reads that is not a distribution (NaN,
 * +inf, no finite entry), makes sequence b -1.  The walk decides in fp32 and marks the
 * sequences where one decision came within a few fp32 errors of flipping; two more kernels
 * walk every marked one again in double-float arithmetic and rewrite its outputs, so the
 * result is the exact rule's except where a decision is closer than ~1e-12 to its boundary
 * (spec_verify_status_offset).  Workspace: spec_verify_workspace_size(SV_MODE_TREE_SAMPLE,
 * B, N, V, dtype) bytes, about 128 V min(N, 8) bytes: the first eight marked sequences get
 * the double-float exponentials of up to 8 reached nodes from the whole grid (115 MB at
 * N = 64, V = 128256 with max_depth = 6 needing 7 of the 8 positions; the size assumes 8);
 * those of them marked only at the final draw (the path certain) have the rejections at
 * the reached node and the draw redone by the same grid, one grid-wide pass per rejection;
 * eight clusters re-walk the others, later ones computing the exponentials in the cluster.
 */
sv_status spec_verify_tree_sample(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, const void *draft_logits,
                                  int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype,
                                  int B, int N, int V, const int32_t *parent,
                                  const int32_t *node_tokens, int max_depth, float temperature,
                                  uint64_t seed, uint64_t offset, int without_replacement,
                                  int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * LAZY verification: the same rules, reading only the rows that can change the result.
 * The rows after the first rejection, or beside the accepted nodes of a tree, never reach
 * the result; these entries walk the rule and read the rows it needs as it goes.  They
 * return exactly what the full entries return whenever every row is a distribution
 * (sampling) or NaN-free (greedy); a bad row the walk never reads does not invalidate the
 * sequence.  Outputs, arguments and errors as the full entries.
 *
 *   spec_verify_sample_lazy       the chain rule of spec_verify_sample, walked level by
 *                                 level over the whole GPU: at level i every sequence still
 *                                 walking streams its target row i and draft row i (one
 *                                 contiguous range of tiles per CTA), the CTA that completes
 *                                 a sequence takes its accept test, and a grid barrier ends
 *                                 the level (several levels at once when the rows of
 *                                 sequences that will have stopped cost less than a level of
 *                                 its own).  The residual masses and the draw, with the
 *                                 double-float re-draw of every marked sequence, are
 *                                 spec_verify_sample's kernels.  Workspace:
 *                                 spec_verify_workspace_size(SV_MODE_SAMPLE_LAZY, B, gamma,
 *                                 V, dtype) bytes.
 *   spec_verify_greedy_lazy       the rule of spec_verify_greedy; no workspace.
 *   spec_verify_tree_greedy_lazy  the rule of spec_verify_tree_greedy (every accepted node's
 *                                 row is read, so the deepest-node rule is unchanged); no
 *                                 workspace.  Both greedy walks give a sequence a cluster of
 *                                 up to 8 CTAs while the batch leaves SMs free (one CTA
 *                                 otherwise), each CTA reading its share of a row's tiles.
 */
sv_status spec_verify_sample_lazy(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, const void *draft_logits,
                                  int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype,
                                  int B, int gamma, int V, const int32_t *draft_tokens,
                                  float temperature, uint64_t seed, uint64_t offset,
                                  int32_t *accepted_len, int32_t *out_tokens, void *workspace,
                                  size_t workspace_bytes, void *stream);
sv_status spec_verify_greedy_lazy(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, sv_dtype dtype, int B, int gamma, int V,
                                  const int32_t *draft_tokens, int32_t *accepted_len,
                                  int32_t *out_tokens, void *stream);
sv_status spec_verify_tree_greedy_lazy(const void *target_logits, int64_t t_batch_stride,
                                       int64_t t_row_stride, sv_dtype dtype, int B, int N, int V,
                                       const int32_t *parent, const int32_t *node_tokens,
                                       int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                                       int32_t *out_path, void *stream);

/*
 * TYPICAL ACCEPTANCE (Medusa's relaxed rule) [SD the Medusa paragraph and the closing note
 * on typical acceptance: accept a draft whose target probability exceeds a threshold that
 * scales with the step's entropy; not distribution-preserving].  The pages give no form
 * or constants; this entry takes
 *   p_i = softmax(t_i / T),  H_i = -sum_j p_i(j) ln p_i(j),  tau_i = min(epsilon, delta e^-H_i),
 * accepts draft x_i while p_i(x_i) > tau_i (left to right), and draws the token at the
 * first failure k (or the bonus at k = gamma) from p_k itself by the inverse CDF with
 * u' = U(b, k, purpose 1) as spec_verify_sample does.
 *   target_logits  [B][gamma+1][V]  as spec_verify_sample (no draft logits are read).
 *   draft_tokens   [B][gamma] int32 (may be NULL when gamma == 0).
 *   temperature > 0; epsilon >= 0, delta >= 0 finite (epsilon = 0 accepts every draft the
 *   target gives positive probability).
 * Outputs as spec_verify_sample.  Rows are read lazily by the level walk of
 * spec_verify_sample_lazy (each tile also sums the entropy's Z): rows 0 .. k only; a token
 * outside [0, V) or a row read that is not a distribution gives -1.  The accept tests are
 * taken in fp32; the final draw is spec_verify_sample's, and every draw whose threshold
 * lies within the fp32 error of a CDF boundary is redone in double-float arithmetic
 * (spec_verify_status_offset with SV_MODE_TYPICAL reports them).  Workspace:
 * spec_verify_workspace_size(SV_MODE_TYPICAL, B, gamma, V, dtype) bytes.
 */
sv_status spec_verify_typical(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                              sv_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens,
                              float temperature, float epsilon, float delta, uint64_t seed,
                              uint64_t offset, int32_t *accepted_len, int32_t *out_tokens,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * SAMPLING verification against a ONE-HOT draft distribution: the drafter proposed x_i
 * with q_i(x_i) = 1 (a prompt-lookup / n-gram drafter, spec_ngram_draft).  The rule of
 * spec_verify_sample with that q [SD "The rule"; the one-hot case of the chain]: accept x_i
 * iff u_i < p_i(x_i) (u_i = U(b, i, purpose 0)); at the first rejection k the residual
 * (p_k - q_k)+ is p_k without x_k, from which the final token is drawn (u' = U(b, k,
 * purpose 1)); the bonus from p_gamma when every draft is accepted.  It equals
 * spec_verify_sample given draft rows that are -inf except 0 at x_i, without those rows.
 *   target_logits  [B][gamma+1][V] as spec_verify_sample; draft_tokens [B][gamma] (may be
 *                  NULL when gamma == 0); temperature > 0 (applied to p).
 * Outputs, errors and the lazy row reads as spec_verify_typical (the level walk, rows
 * 0 .. k; near-boundary accept tests and final draws redone in double-float).  Workspace:
 * spec_verify_workspace_size(SV_MODE_SAMPLE_ONEHOT, B, gamma, V, dtype) bytes.
 */
sv_status spec_verify_sample_onehot(const void *target_logits, int64_t t_batch_stride,
                                    int64_t t_row_stride, sv_dtype dtype, int B, int gamma, int V,
                                    const int32_t *draft_tokens, float temperature, uint64_t seed,
                                    uint64_t offset, int32_t *accepted_len, int32_t *out_tokens,
                                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Prompt-lookup (n-gram) drafting [MS lookup_draft; SD Exercise 4 ngram_draft]: the drafts
 * that the verification entries take, from the token history itself.
 *
 *   history  [B][stride] int32   each sequence's tokens so far, lengths[b] of them valid
 *                                (a length outside [0, stride] is clamped to it).
 *   n        1 .. 64             the n-gram: the sequence's last n tokens (the tail).
 *   k        0 .. SV_MAX_GAMMA   tokens to propose.
 *   pad      nonzero: always propose k tokens, filling with the last token (Exercise 4).
 * The drafts are the tokens that followed the tail's most recent earlier occurrence (a
 * start i <= len - n - 1 whose n tokens equal the tail), at most k of them; none without a
 * match (or with len < n + 1) unless padded.  Outputs: drafts [B][k] (-1 in unused slots),
 * count [B].  The drafter's q is one-hot on each draft: verify with spec_verify_greedy or
 * spec_verify_sample_onehot.
 * No workspace; one CTA per sequence searches from the end of the history backwards.
 */
sv_status spec_ngram_draft(const int32_t *history, int64_t stride, const int32_t *lengths, int B, int n,
                           int k, int pad, int32_t *drafts, int32_t *count, void *stream);

/*
 * Greedy verification that allocates nothing and takes no workspace.  (The pages have no
 * counterpart: this is a deployment variant of spec_verify_greedy.)
 *
 * For callers that cannot hand the library device memory -- code running inside another
 * runtime's execution step whose framework owns every buffer, or a serving loop that must
 * not call cudaMalloc once it is running.  Same arguments, rules and results as
 * spec_verify_greedy, minus the workspace: the per-tile maxima live in a fixed,
 * 256-byte-aligned device array of SV_NOALLOC_SCRATCH_BYTES that is part of the library and
 * stays resident on every GPU that loads it until the process exits.
 *   - Limit: B * (gamma + 1) * ceil(V / tile) * 4 <= SV_NOALLOC_SCRATCH_BYTES, with tile =
 *     2048 logits for bf16 and 1024 for fp32 (4 MiB covers, e.g., B = 512, gamma = 6,
 *     V = 152064 bf16: 1.1 MB).  Larger problems return SV_ERR_WORKSPACE before anything is
 *     enqueued.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - All calls on a device share the array.  Calls whose kernels overlap on the GPU (for
 *     example on two streams) race on it; the caller must order them.
 *   - It calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define SV_NOALLOC_SCRATCH_BYTES (4u << 20)
sv_status spec_verify_greedy_noalloc(const void *target_logits, int64_t t_batch_stride,
                                     int64_t t_row_stride, sv_dtype dtype, int B, int gamma,
                                     int V, const int32_t *draft_tokens, int32_t *accepted_len,
                                     int32_t *out_tokens, void *stream);

/*
 * Test hook: the per-row statistics of the sampling path [SD apply_temperature].
 *   logits [B][rows_per_seq][V].  m_out[b*rows_per_seq + r] = max_j l_j / T,
 *   lse_out[...] = m + ln sum_j exp(l_j / T - m); both NaN for a row with a NaN, a +inf or
 *   no finite entry.  Computed by the same kernels as spec_verify_sample.
 */
sv_status spec_verify_row_stats(const void *logits, int64_t batch_stride, int64_t row_stride,
                                sv_dtype dtype, int B, int rows_per_seq, int V,
                                float temperature, float *m_out, float *lse_out,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * Test hook: the uniforms the sampler draws.  out[b * positions + i] = u(b, i, purpose) as
 * defined under spec_verify_sample, for b < B, i < positions, purpose in {0, 1}.
 */
sv_status spec_verify_uniforms(uint64_t seed, uint64_t offset, int B, int positions,
                               int purpose, float *out, void *stream);

/*
 * Where a sampling call keeps its device-side outcome inside its workspace: the byte offset
 * of an int32 array ((size_t)-1 for a mode without one -- greedy, tree greedy, row
 * statistics -- or bad sizes).  Modes and rows as spec_verify_workspace_size:
 * SV_MODE_SAMPLE, SV_MODE_TREE_SAMPLE, SV_MODE_SAMPLE_LAZY, SV_MODE_TYPICAL and
 * SV_MODE_SAMPLE_ONEHOT.  Read it after the call's stream has completed:
 *   [0]      sequences the call marked: an fp32 decision near enough to its boundary to be
 *            in doubt -- an accept test with |u q - p| below 1e-6 of max(p, u q) (plus, for
 *            the tree walk, the size of p's terms), a draw whose threshold lies within a few
 *            1e-8 .. 1e-6 of the draw's total mass from a CDF boundary, a residual mass or a
 *            remaining q mass too small to trust, or a rounding fallback ("The rule";
 *            readings R2, R3, R14);
 *   [3]      SV_OK, or SV_ERR_TIMEOUT if a bounded wait of the chain re-draw gave up (2 s:
 *            only when the GPU cannot hold its grid, e.g. another kernel holds every SM) --
 *            the sequences it did not finish keep their fp32 result;
 *   [4]      sequences redone in double-float arithmetic (equal to [0] unless [3] is set);
 *   [8 + b]  nonzero if sequence b was marked.
 */
size_t spec_verify_status_offset(sv_mode mode, int B, int rows, int V, sv_dtype dtype);

/*
 * Test hook of the library's software waits (the chain re-draw's bounded wait for a flag
 * another warp sets, and the bounded grid barrier): one CTA waits for a flag and then meets
 * the barrier expecting expected_arrivals (1 or 2) CTAs.  With 1 the CTA sets the flag
 * itself and passes both at once (ctl[3] = 0).  With 2 nobody sets the flag and nobody
 * else arrives: each wait gives up after limit_us (at most 5 s) and SV_ERR_TIMEOUT is
 * written to ctl[3].  ctl: a device int32 array of 8 the call overwrites.  The kernel
 * returns either way, so the context stays usable.
 */
sv_status spec_verify_wait_selftest(int *ctl, int expected_arrivals, uint32_t limit_us, void *stream);

/*
 * Test hook: exp(y_hi[i] + y_lo[i]) for arguments <= 0 in the double-float arithmetic of
 * the re-draw (result hi + lo, about 48 significant bits; 0 below -87).  Device arrays of n.
 */
sv_status spec_verify_exp_df(const float *y_hi, const float *y_lo, int n, float *out_hi, float *out_lo,
                             void *stream);

/*
 * Optional timing instrumentation for the CALLING THREAD (the only state the library
 * keeps, and it is thread-local).  With events != NULL, each later call of
 * spec_verify_sample / _greedy / _greedy_noalloc / _tree_greedy / _tree_sample / _sample_lazy /
 * _typical / _sample_onehot on this thread
 * records events[0] on its stream before its first kernel and events[s] after its s-th
 * kernel (s = 1 .. n_events-1; sampling has 4 kernels: row statistics, decide, residual
 * masses, and the inverse-CDF draw with the extended-precision re-draw of near-boundary
 * sequences (one cooperative grid); a sampling call with B = 1 and (2 gamma + 1) row tiles
 * of at most 256 runs all four stages in one kernel of one thread block, and records
 * events[2..4] right after it; greedy and tree have 2: tile maxima, finalize; the lazy
 * greedy walks have 1; tree sampling has 3: the walk, the re-walk's exponentials with
 * the final re-draw of the sequences marked only at their final draw, the re-walk; lazy sampling has 3: the level walk, residual masses, the draw with its re-draw;
 * typical acceptance and one-hot sampling have 2: the level walk, the draw with its
 * re-draw).  The events are cudaEvent_t handles created and owned by the caller; recording
 * them adds no synchronisation.  Pass NULL (or 0) to turn it off.
 * Returns SV_ERR_INVALID_ARG for n_events < 0 or > 8.
 */
sv_status spec_verify_set_stage_events(void *const *events, int n_events);

/*
 * The bounds-checked build (the library compiled with -DSV_CHECKS; a debugging aid, not the
 * product build).  Its kernels check every index into the buffers the library sizes itself
 * -- the workspace regions (tile partials, row statistics, plans, residual masses, re-draw
 * records and unit sums, level lists and counters), tile and unit counts, tree node ids,
 * n-gram positions and the rows of accepted_len / out_tokens -- against the extent the
 * library knows, skip an access outside it and record the first such violation in a
 * device-side word.  This call waits for the current device, copies that word into info
 * (may be NULL): info[0] = site (a 16-bit tag of the source file's name << 16 | line),
 * info[1] = the offending index, info[2] = the extent (both clamped to int32), info[3] =
 * the number of violations; then clears it.  Returns SV_OK when nothing was recorded,
 * SV_ERR_CHECK when something was, SV_ERR_CUDA if the copy failed, and SV_ERR_UNSUPPORTED
 * (info zeroed) in the normal build.
 */
sv_status spec_verify_check_word(int32_t *info);
/* Test hook of the bounds-checked build: one kernel that checks `index` against `extent`
 * (and accesses no memory), so that a test can see a violation recorded and reported by
 * spec_verify_check_word.  SV_ERR_UNSUPPORTED in the normal build. */
sv_status spec_verify_check_selftest(int64_t index, int64_t extent);

/* A static, human-readable name for a status code. */
const char *spec_verify_status_string(sv_status status);

/* ABI version of this header (major * 100 + minor). */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
