// sv_api.cu -- the C ABI of libspecverify: argument checks, workspace layout and the
// launch sequence of each entry point.  Every check happens before the first launch, so
// an error return means nothing was enqueued.
#include <cmath>
#include <cstdint>

#include "spec_verify.h"
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace {

using sv::Logits;

constexpr int64_t kMaxGrid = 0x7FFFFFFF;

using sv::ntile_of;
using sv::vec_ok;

bool dtype_ok(sv_dtype d) { return d == SV_FP32 || d == SV_BF16; }
int res_tile_elems(sv_dtype d) {
    return d == SV_BF16 ? sv::res_tile_elems<sv::BF16>() : sv::res_tile_elems<sv::F32>();
}
int nrt_of(int V, sv_dtype d) { return int((int64_t(V) + res_tile_elems(d) - 1) / res_tile_elems(d)); }
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t partial = 0, rowstat = 0, plan = 0, csum = 0;
    size_t rctl = 0, rbar = 0, rlist = 0, rsum = 0, ramb = 0, rresc = 0;  // re-draw: control + marks, barrier, records, scratch
    size_t rec = 0, et = 0, us = 0, npos = 0, um = 0, pmax = 0, pcnt = 0;  // re-walk (tree sampling; rctl, rsum too)
    size_t zpart = 0, xval = 0, lctl = 0, lact = 0, tcnt = 0, lstate = 0, lavail = 0;  // the level walks
    size_t total = 0;
};

// Workspace regions (each 256-byte aligned):
//   partial  per (row, 4 KB tile): float2 (M, S) for sampling / row stats, the float
//            maximum for greedy / tree;
//   rowstat  per row: float2 (M, S)                             (sampling only)
//   plan     per sequence: int2 (stop row k, mode)              (sampling only)
//   csum     per (sequence, 2 KB residual tile): residual mass  (sampling only)
//   rctl     the re-draw's control words, then the per-sequence marks rflag[B];
//   rbar     the words of the re-draw's grid barrier;
//   rlist    2 B RefineInfo records (main list, rescan list);
//   rsum, ramb, rresc  the re-draw's scratch: per main-list sequence 5 x refine_units(V)
//            double-float unit sums and refine_units(V) near-logit counts; kRescanChunk x
//            (2 gamma + 1) x refine_units(V) unit sums for the rescan list (sampling only; see
//            sv_internal.h): the re-draw of every near-boundary sequence
// Tree sampling and lazy sampling: the walk's unit masses (partial) and per-CTA row
// statistics (rowstat), then the re-walk's control block, marks and record lengths (rctl),
// records (rec), stored exponentials and their unit sums (et, us), support counts (npos),
// unit masses (um), per-CTA sums (rsum), maxima (pmax) and counts (pcnt); see
// sv_internal.h.  The exponentials dominate: 16 V bytes per recorded node and listed
// sequence.
// Recorded positions of the tree-sampling walk: max_depth + 1 <= N (tree) or gamma + 1
// (lazy chain), at most kTreeRecNodes.
int rec_positions(sv_mode mode, int rows) {
    return mode == SV_MODE_TREE_SAMPLE ? (rows < sv::kTreeRecNodes ? rows : sv::kTreeRecNodes)
                                       : sv::tree_rec_nodes(rows);
}

Layout layout(sv_mode mode, int B, int rows, int V, sv_dtype dtype) {
    Layout L;
    if (B <= 0 || V <= 0 || rows < 0 || !dtype_ok(dtype)) return L;
    const size_t ntile = size_t(ntile_of(V, dtype));
    size_t R = 0;
    switch (mode) {
    case SV_MODE_SAMPLE:
    case SV_MODE_SAMPLE_LAZY: R = size_t(2) * rows + 1; break;
    case SV_MODE_TYPICAL:
    case SV_MODE_SAMPLE_ONEHOT: R = size_t(rows) + 1; break;
    case SV_MODE_GREEDY: R = size_t(rows) + 1; break;
    case SV_MODE_TREE:
    case SV_MODE_ROW_STATS: R = size_t(rows); break;
    case SV_MODE_TREE_SAMPLE: {
        L.partial = 0;
        size_t off = up256(size_t(B) * size_t(nrt_of(V, dtype)) * 4);
        L.rowstat = off;
        off += up256(size_t(B) * sv::kTreeSampleCluster * 2 * 8);
        const size_t K = size_t(rec_positions(mode, rows));
        const size_t nu = size_t(sv::tree_refine_units(V)), S = sv::kMaxTreeRefine, C = sv::kTreeRefineCluster;
        L.rctl = off;
        off += up256((size_t(sv::kTrCtlWords) + 2 * size_t(B)) * 4);
        L.rec = off;
        off += up256(size_t(B) * K * 16);
        L.et = off;
        off += up256(S * K * 2 * size_t(V) * 8);
        L.us = off;
        off += up256(S * K * 2 * nu * 8);
        L.npos = off;
        off += up256(S * K * 4);
        L.um = off;
        off += up256(2 * S * nu * 8);
        L.rsum = off;
        off += up256(S * 2 * C * 2 * 8);
        L.pmax = off;
        off += up256(S * C * 2 * 4);
        L.pcnt = off;
        off += up256(S * C * 4);
        L.total = off;
        return L;
    }
    default: return L;
    }
    L.partial = 0;
    size_t off = up256(size_t(B) * R * ntile * 8);
    const bool sampling = mode == SV_MODE_SAMPLE || mode == SV_MODE_SAMPLE_LAZY || mode == SV_MODE_TYPICAL ||
                          mode == SV_MODE_SAMPLE_ONEHOT;
    if (sampling) {
        L.rowstat = off;
        off += up256(size_t(B) * R * 8);
        L.plan = off;
        off += up256(size_t(B) * 8);
        L.csum = off;
        off += up256(size_t(B) * size_t(nrt_of(V, dtype)) * 4);
        L.rctl = off;
        off += up256((size_t(sv::kRefineCtlWords) + size_t(B)) * 4);
        L.rbar = off;
        off += up256(size_t(sv::kRefineCtlWords) * 4);
        L.rlist = off;
        off += up256(size_t(2) * B * sizeof(sv::RefineInfo));
        const size_t nu = size_t(sv::refine_units(V));
        L.rsum = off;
        off += up256(size_t(B) * 5 * nu * 8);
        L.ramb = off;
        off += up256(size_t(B) * nu * 4);
        L.rresc = off;
        off += up256(size_t(sv::kRescanChunk) * R * nu * 8);
    }
    if (sampling && mode != SV_MODE_SAMPLE) {  // the level walk's own words
        if (mode == SV_MODE_TYPICAL) {
            L.zpart = off;
            off += up256(size_t(B) * R * ntile * 4);
        }
        L.xval = off;
        off += up256(size_t(B) * R * 4);
        L.lctl = off;
        off += up256((size_t(8) + rows + 2) * 4);
        L.lact = off;
        off += up256(size_t(2) * B * 4);
        L.tcnt = off;
        off += up256(size_t(B) * 4);
        L.lstate = off;
        off += up256(size_t(B) * 4);
        L.lavail = off;
        off += up256(size_t(B) * 4);
    }
    L.total = off;
    return L;
}

sv_status check_workspace(const Layout &L, void *ws, size_t bytes) {
    if (L.total == 0) return SV_OK;
    if (ws == nullptr || bytes < L.total || reinterpret_cast<uintptr_t>(ws) % 16 != 0)
        return SV_ERR_WORKSPACE;
    return SV_OK;
}

char *at(void *ws, size_t off) { return static_cast<char *>(ws) + off; }

sv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

sv::TreeRefineWs tree_refine_ws(const Layout &L, void *ws, int B) {
    sv::TreeRefineWs r;
    r.ctl = reinterpret_cast<int *>(at(ws, L.rctl));
    r.mark = r.ctl + sv::kTrCtlWords;
    r.rlen = r.mark + B;
    r.rec = reinterpret_cast<float4 *>(at(ws, L.rec));
    r.et = reinterpret_cast<sv::df *>(at(ws, L.et));
    r.us = reinterpret_cast<sv::df *>(at(ws, L.us));
    r.npos = reinterpret_cast<int *>(at(ws, L.npos));
    r.um = reinterpret_cast<sv::df *>(at(ws, L.um));
    r.part = reinterpret_cast<sv::df *>(at(ws, L.rsum));
    r.pmax = reinterpret_cast<float *>(at(ws, L.pmax));
    r.pcnt = reinterpret_cast<int *>(at(ws, L.pcnt));
    return r;
}

// Tile counts (and every partial index) stay below 2^31.
bool tiles_fit(int B, int64_t R, int ntile) { return int64_t(B) * R * ntile <= kMaxGrid; }

// Optional per-thread timing events (spec_verify_set_stage_events).
constexpr int kMaxStageEvents = 8;
thread_local cudaEvent_t t_events[kMaxStageEvents];
thread_local int t_nevents = 0;

cudaError_t mark(int s, cudaStream_t stream) { return sv::mark_stage(s, stream); }

}  // namespace

namespace {
// The lazy walks of the sampling chain, of a one-hot q and of typical acceptance: the level
// kernel reads rows 0 .. k of each sequence and plans its draw; then (the chain only) the
// residual masses of the stop rows; then the draw with the double-float re-draw of every
// near-boundary sequence.  Arguments already checked, except the workspace.
sv_status level_walk(int rule, sv_mode mode, const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                     const void *draft_logits, int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype, int B,
                     int gamma, int V, const int32_t *draft_tokens, float temperature, float epsilon, float delta,
                     uint64_t seed, uint64_t offset, int32_t *accepted_len, int32_t *out_tokens, void *workspace,
                     size_t workspace_bytes, void *stream) {
    const Layout L = layout(mode, B, gamma, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;
    const bool chain = rule == sv::kRuleSample;
    const int ntile = ntile_of(V, dtype), nrt = nrt_of(V, dtype);
    if (!tiles_fit(B, chain ? 2 * int64_t(gamma) + 1 : int64_t(gamma) + 1, ntile)) return SV_ERR_INVALID_ARG;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype) &&
                     (!chain || gamma == 0 || vec_ok(draft_logits, d_batch_stride, d_row_stride, dtype));
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    const Logits d{chain && gamma > 0 ? draft_logits : target_logits, d_batch_stride, d_row_stride};
    const float c = float(1.4426950408889634 / double(temperature));  // log2(e) / T
    const int dt = dtype == SV_BF16 ? 1 : 0;
    const int R = chain ? 2 * gamma + 1 : gamma + 1;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *rctl = reinterpret_cast<int *>(at(workspace, L.rctl));
    int *rbar = reinterpret_cast<int *>(at(workspace, L.rbar));
    int *lavail = reinterpret_cast<int *>(at(workspace, L.lavail));
    sv::LevelArgs la;
    la.t = t;
    la.d = d;
    la.B = B;
    la.gamma = gamma;
    la.V = V;
    la.ntile = ntile;
    la.R = R;
    la.c = c;
    la.x = draft_tokens;
    la.seed = seed;
    la.offset = offset;
    la.epsilon = epsilon;
    la.delta = delta;
    la.partial = reinterpret_cast<float2 *>(at(workspace, L.partial));
    la.zpart = reinterpret_cast<float *>(at(workspace, L.zpart));
    la.xval = reinterpret_cast<float *>(at(workspace, L.xval));
    la.rowstat = reinterpret_cast<float2 *>(at(workspace, L.rowstat));
    la.plan = reinterpret_cast<int2 *>(at(workspace, L.plan));
    la.accepted_len = accepted_len;
    la.out_tokens = out_tokens;
    la.rctl = rctl;
    la.rbar = rbar;
    la.lctl = reinterpret_cast<int *>(at(workspace, L.lctl));
    la.lact = reinterpret_cast<int *>(at(workspace, L.lact));
    la.tcnt = reinterpret_cast<int *>(at(workspace, L.tcnt));
    la.lstate = reinterpret_cast<int *>(at(workspace, L.lstate));
    la.lavail = lavail;
    float *csum = reinterpret_cast<float *>(at(workspace, L.csum));
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess) e = sv::launch_level(rule, dt, vec, la, s);
    if (e == cudaSuccess) e = mark(1, s);
    int st = 2;
    if (e == cudaSuccess && chain && gamma > 0) {
        e = sv::launch_residual_tiles(dt, vec, t, d, B, gamma, V, nrt, c, la.rowstat, la.plan, csum, s);
        if (e == cudaSuccess) e = mark(st++, s);
    }
    if (e == cudaSuccess)
        e = sv::launch_draw_refine(dt, vec, t, d, B, gamma, V, ntile, nrt, c, temperature, seed, offset, rule, R, lavail,
                                   draft_tokens, la.partial, la.rowstat, la.plan, csum, accepted_len, out_tokens, rctl,
                                   rbar, reinterpret_cast<sv::RefineInfo *>(at(workspace, L.rlist)),
                                   at(workspace, L.rsum), reinterpret_cast<int *>(at(workspace, L.ramb)),
                                   at(workspace, L.rresc), chain && gamma > 0, s);
    if (e == cudaSuccess) e = mark(st, s);
    return cuda_status(e);
}
}  // namespace

#ifdef SV_CHECKS
namespace sv {
__device__ int g_check[4];
__device__ bool check_fail(uint32_t site, int64_t idx, int64_t n) {
    auto clamp32 = [](int64_t v) { return int(v > 0x7FFFFFFF ? 0x7FFFFFFF : (v < -0x7FFFFFFF ? -0x7FFFFFFF : v)); };
    if (atomicCAS(&g_check[0], 0, int(site)) == 0) {
        g_check[1] = clamp32(idx);
        g_check[2] = clamp32(n);
    }
    atomicAdd(&g_check[3], 1);
    return false;
}
// One check of `index` against `extent` and nothing else (no memory is accessed).
__global__ void check_selftest_kernel(int64_t index, int64_t extent) {
    if (threadIdx.x == 0) (void)SV_IN(index, extent);
}
}  // namespace sv
#endif

namespace sv {
cudaError_t mark_stage(int s, cudaStream_t stream) {
    if (s < t_nevents && t_events[s] != nullptr) return cudaEventRecord(t_events[s], stream);
    return cudaSuccess;
}
}  // namespace sv

extern "C" {

int spec_verify_version(void) { return 100; }

sv_status spec_verify_check_word(int32_t *info) {
#ifdef SV_CHECKS
    int h[4] = {0, 0, 0, 0};
    const int z[4] = {0, 0, 0, 0};
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpyFromSymbol(h, sv::g_check, sizeof(h)) != cudaSuccess ||
        cudaMemcpyToSymbol(sv::g_check, z, sizeof(z)) != cudaSuccess)
        return SV_ERR_CUDA;
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = h[i];
    return h[0] != 0 ? SV_ERR_CHECK : SV_OK;
#else
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = 0;
    return SV_ERR_UNSUPPORTED;
#endif
}

sv_status spec_verify_check_selftest(int64_t index, int64_t extent) {
#ifdef SV_CHECKS
    sv::check_selftest_kernel<<<1, 32>>>(index, extent);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
#else
    (void)index;
    (void)extent;
    return SV_ERR_UNSUPPORTED;
#endif
}

const char *spec_verify_status_string(sv_status s) {
    switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported dtype or mode";
    case SV_ERR_CUDA: return "CUDA launch failed";
    case SV_ERR_TIMEOUT: return "a bounded device wait gave up";
    case SV_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case SV_ERR_CHECK: return "an internal index left its extent (bounds-checked build)";
    }
    return "unknown status";
}

size_t spec_verify_workspace_size(sv_mode mode, int B, int rows, int V, sv_dtype dtype) {
    return layout(mode, B, rows, V, dtype).total;
}

sv_status spec_verify_sample(const void *target_logits, int64_t t_batch_stride,
                             int64_t t_row_stride, const void *draft_logits,
                             int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype, int B,
                             int gamma, int V, const int32_t *draft_tokens, float temperature,
                             uint64_t seed, uint64_t offset, int32_t *accepted_len,
                             int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (t_batch_stride < 0 || t_row_stride < 0 || d_batch_stride < 0 || d_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens) return SV_ERR_INVALID_ARG;
    if (gamma > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_INVALID_ARG;
    const int ntile = ntile_of(V, dtype), nrt = nrt_of(V, dtype);
    const int R = 2 * gamma + 1;
    if (!tiles_fit(B, R, ntile)) return SV_ERR_INVALID_ARG;
    const Layout L = layout(SV_MODE_SAMPLE, B, gamma, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;

    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype) &&
                     (gamma == 0 || vec_ok(draft_logits, d_batch_stride, d_row_stride, dtype));
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    const Logits d{gamma > 0 ? draft_logits : target_logits, d_batch_stride, d_row_stride};
    const float c = float(1.4426950408889634 / double(temperature));  // log2(e) / T
    const int dt = dtype == SV_BF16 ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *partial = at(workspace, L.partial), *rowstat = at(workspace, L.rowstat);
    void *plan = at(workspace, L.plan);
    float *csum = reinterpret_cast<float *>(at(workspace, L.csum));

    cudaError_t e = mark(0, s);
    if (sv::single_sample_fits(B, gamma, ntile)) {  // one kernel; every later stage event after it
        if (e == cudaSuccess)
            e = sv::launch_single_sample(dt, vec, t, d, gamma, V, ntile, nrt, c, temperature, seed, offset, draft_tokens,
                                         partial, rowstat, plan, csum, accepted_len, out_tokens,
                                         reinterpret_cast<int *>(at(workspace, L.rctl)),
                                         reinterpret_cast<int *>(at(workspace, L.rbar)),
                                         reinterpret_cast<sv::RefineInfo *>(at(workspace, L.rlist)),
                                         at(workspace, L.rsum), reinterpret_cast<int *>(at(workspace, L.ramb)),
                                         at(workspace, L.rresc), s);
        for (int st = 1; st <= 4 && e == cudaSuccess; ++st) e = mark(st, s);
        return cuda_status(e);
    }
    if (e == cudaSuccess)
        e = sv::launch_stats_tiles(dt, vec, t, gamma + 1, d, R, B, V, ntile, c, partial, s);
    if (e == cudaSuccess) e = mark(1, s);
    int *rctl = reinterpret_cast<int *>(at(workspace, L.rctl));
    int *rflag = rctl + sv::kRefineCtlWords;
    int *rbar = reinterpret_cast<int *>(at(workspace, L.rbar));
    sv::RefineInfo *rinfo = reinterpret_cast<sv::RefineInfo *>(at(workspace, L.rlist));
    if (e == cudaSuccess)
        e = sv::launch_decide(dt, t, d, B, gamma, V, ntile, c, draft_tokens, seed, offset, partial,
                              rowstat, plan, accepted_len, out_tokens, rflag, rctl, rbar, s);
    if (e == cudaSuccess) e = mark(2, s);
    if (e == cudaSuccess && gamma > 0)
        e = sv::launch_residual_tiles(dt, vec, t, d, B, gamma, V, nrt, c, rowstat, plan, csum, s);
    if (e == cudaSuccess) e = mark(3, s);
    if (e == cudaSuccess)
        e = sv::launch_draw_refine(dt, vec, t, d, B, gamma, V, ntile, nrt, c, temperature, seed, offset,
                                   sv::kRuleSample, R, nullptr, draft_tokens, partial, rowstat, plan, csum, accepted_len,
                                   out_tokens, rctl, rbar, rinfo,
                                   at(workspace, L.rsum), reinterpret_cast<int *>(at(workspace, L.ramb)),
                                   at(workspace, L.rresc), gamma > 0, s);
    if (e == cudaSuccess) e = mark(4, s);
    return cuda_status(e);
}

sv_status spec_verify_greedy(const void *target_logits, int64_t t_batch_stride,
                             int64_t t_row_stride, sv_dtype dtype, int B, int gamma, int V,
                             const int32_t *draft_tokens, int32_t *accepted_len,
                             int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (t_batch_stride < 0 || t_row_stride < 0) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens || (gamma > 0 && !draft_tokens))
        return SV_ERR_INVALID_ARG;
    const int ntile = ntile_of(V, dtype);
    if (!tiles_fit(B, gamma + 1, ntile)) return SV_ERR_INVALID_ARG;
    const Layout L = layout(SV_MODE_GREEDY, B, gamma, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype);
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *partial = at(workspace, L.partial);
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess)
        e = sv::launch_max_tiles(dtype == SV_BF16, vec, t, gamma + 1, B, V, ntile, partial, s);
    if (e == cudaSuccess) e = mark(1, s);
    if (e == cudaSuccess)
        e = sv::launch_greedy_finalize(dtype == SV_BF16, vec, t, B, gamma, V, ntile, partial, draft_tokens,
                                       accepted_len,
                                       out_tokens, s);
    if (e == cudaSuccess) e = mark(2, s);
    return cuda_status(e);
}

sv_status spec_verify_tree_greedy(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, sv_dtype dtype, int B, int N, int V,
                                  const int32_t *parent, const int32_t *node_tokens,
                                  int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                                  int32_t *out_path, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (max_depth < 0 || max_depth >= N || t_batch_stride < 0 || t_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !parent || !node_tokens || !accepted_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    const int ntile = ntile_of(V, dtype);
    if (!tiles_fit(B, N, ntile)) return SV_ERR_INVALID_ARG;
    const Layout L = layout(SV_MODE_TREE, B, N, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype);
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *partial = at(workspace, L.partial);
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess)
        e = sv::launch_max_tiles(dtype == SV_BF16, vec, t, N, B, V, ntile, partial, s);
    if (e == cudaSuccess) e = mark(1, s);
    if (e == cudaSuccess)
        e = sv::launch_tree_finalize(dtype == SV_BF16, vec, t, B, N, V, ntile, partial, parent, node_tokens,
                                     max_depth,
                                     accepted_len, out_tokens, out_path, s);
    if (e == cudaSuccess) e = mark(2, s);
    return cuda_status(e);
}

sv_status spec_verify_tree_sample(const void *target_logits, int64_t t_batch_stride,
                                  int64_t t_row_stride, const void *draft_logits,
                                  int64_t d_batch_stride, int64_t d_row_stride, sv_dtype dtype,
                                  int B, int N, int V, const int32_t *parent,
                                  const int32_t *node_tokens, int max_depth, float temperature,
                                  uint64_t seed, uint64_t offset, int without_replacement,
                                  int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (max_depth < 0 || max_depth >= N || t_batch_stride < 0 || t_row_stride < 0 || d_batch_stride < 0 ||
        d_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !draft_logits || !parent || !node_tokens || !accepted_len || !out_tokens)
        return SV_ERR_INVALID_ARG;
    const Layout L = layout(SV_MODE_TREE_SAMPLE, B, N, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype) &&
                     vec_ok(draft_logits, d_batch_stride, d_row_stride, dtype);
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    const Logits d{draft_logits, d_batch_stride, d_row_stride};
    const float c = float(1.4426950408889634 / double(temperature));  // log2(e) / T
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const sv::TreeRefineWs rw = tree_refine_ws(L, workspace, B);
    const int K = sv::tree_rec_nodes(max_depth);
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess)
        e = sv::launch_tree_sample(dtype == SV_BF16, vec, t, d, B, N, V, parent, node_tokens, max_depth, c,
                                   seed, offset, without_replacement, nrt_of(V, dtype),
                                   reinterpret_cast<float *>(at(workspace, 0)),
                                   reinterpret_cast<float2 *>(at(workspace, L.rowstat)), rw, K, accepted_len,
                                   out_tokens, out_path, s);
    if (e == cudaSuccess) e = mark(1, s);
    if (e == cudaSuccess)
        e = sv::launch_tree_exp(dtype == SV_BF16, t, d, B, N, V, parent, node_tokens, max_depth, temperature, seed,
                                offset, without_replacement, K, rw, accepted_len, out_tokens, out_path, s);
    if (e == cudaSuccess) e = mark(2, s);
    if (e == cudaSuccess)
        e = sv::launch_tree_rewalk(dtype == SV_BF16, t, d, B, N, V, parent, node_tokens, max_depth, temperature,
                                   seed, offset, without_replacement, K, rw, accepted_len, out_tokens, out_path, s);
    if (e == cudaSuccess) e = mark(3, s);
    return cuda_status(e);
}

sv_status spec_verify_sample_lazy(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                                  const void *draft_logits, int64_t d_batch_stride, int64_t d_row_stride,
                                  sv_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens,
                                  float temperature, uint64_t seed, uint64_t offset, int32_t *accepted_len,
                                  int32_t *out_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (t_batch_stride < 0 || t_row_stride < 0 || d_batch_stride < 0 || d_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens) return SV_ERR_INVALID_ARG;
    if (gamma > 0 && (!draft_logits || !draft_tokens)) return SV_ERR_INVALID_ARG;
    return level_walk(sv::kRuleSample, SV_MODE_SAMPLE_LAZY, target_logits, t_batch_stride, t_row_stride,
                      draft_logits, d_batch_stride, d_row_stride, dtype, B, gamma, V, draft_tokens, temperature, 0.f,
                      0.f, seed, offset, accepted_len, out_tokens, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {
// The target-only walks: typical acceptance (onehot = 0) or sampling against a one-hot q
// (onehot = 1).
sv_status target_walk(int onehot, const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                      sv_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens, float temperature,
                      float epsilon, float delta, uint64_t seed, uint64_t offset, int32_t *accepted_len,
                      int32_t *out_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB || t_batch_stride < 0 ||
        t_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    if (!(epsilon >= 0.f) || !std::isfinite(epsilon) || !(delta >= 0.f) || !std::isfinite(delta))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
    return level_walk(onehot ? sv::kRuleOnehot : sv::kRuleTypical, onehot ? SV_MODE_SAMPLE_ONEHOT : SV_MODE_TYPICAL,
                      target_logits, t_batch_stride, t_row_stride, nullptr, 0, 0, dtype, B, gamma, V, draft_tokens,
                      temperature, epsilon, delta, seed, offset, accepted_len, out_tokens, workspace, workspace_bytes,
                      stream);
}
}  // namespace

extern "C" {

sv_status spec_verify_typical(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride, sv_dtype dtype,
                              int B, int gamma, int V, const int32_t *draft_tokens, float temperature, float epsilon,
                              float delta, uint64_t seed, uint64_t offset, int32_t *accepted_len,
                              int32_t *out_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    return target_walk(0, target_logits, t_batch_stride, t_row_stride, dtype, B, gamma, V, draft_tokens, temperature,
                       epsilon, delta, seed, offset, accepted_len, out_tokens, workspace, workspace_bytes, stream);
}

sv_status spec_verify_sample_onehot(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                                    sv_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens,
                                    float temperature, uint64_t seed, uint64_t offset, int32_t *accepted_len,
                                    int32_t *out_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    return target_walk(1, target_logits, t_batch_stride, t_row_stride, dtype, B, gamma, V, draft_tokens, temperature,
                       0.f, 0.f, seed, offset, accepted_len, out_tokens, workspace, workspace_bytes, stream);
}

sv_status spec_verify_greedy_lazy(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                                  sv_dtype dtype, int B, int gamma, int V, const int32_t *draft_tokens,
                                  int32_t *accepted_len, int32_t *out_tokens, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB || t_batch_stride < 0 ||
        t_row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens || (gamma > 0 && !draft_tokens)) return SV_ERR_INVALID_ARG;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype);
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess)
        e = sv::launch_greedy_walk(dtype == SV_BF16, vec, t, B, gamma + 1, V, true, nullptr, draft_tokens, gamma,
                                   accepted_len, out_tokens, nullptr, s);
    if (e == cudaSuccess) e = mark(1, s);
    return cuda_status(e);
}

sv_status spec_verify_tree_greedy_lazy(const void *target_logits, int64_t t_batch_stride, int64_t t_row_stride,
                                       sv_dtype dtype, int B, int N, int V, const int32_t *parent,
                                       const int32_t *node_tokens, int max_depth, int32_t *accepted_len,
                                       int32_t *out_tokens, int32_t *out_path, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (max_depth < 0 || max_depth >= N || t_batch_stride < 0 || t_row_stride < 0) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !parent || !node_tokens || !accepted_len || !out_tokens) return SV_ERR_INVALID_ARG;
    const bool vec = vec_ok(target_logits, t_batch_stride, t_row_stride, dtype);
    const Logits t{target_logits, t_batch_stride, t_row_stride};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = mark(0, s);
    if (e == cudaSuccess)
        e = sv::launch_greedy_walk(dtype == SV_BF16, vec, t, B, N, V, false, parent, node_tokens, max_depth,
                                   accepted_len, out_tokens, out_path, s);
    if (e == cudaSuccess) e = mark(1, s);
    return cuda_status(e);
}

sv_status spec_ngram_draft(const int32_t *history, int64_t stride, const int32_t *lengths, int B, int n, int k,
                           int pad, int32_t *drafts, int32_t *count, void *stream) {
    if (B < 0 || n < 1 || n > sv::kMaxNgram || k < 0 || k > SV_MAX_GAMMA || stride < 0 || stride > (1 << 30))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!history || !lengths || !count || (k > 0 && !drafts)) return SV_ERR_INVALID_ARG;
    return cuda_status(sv::launch_ngram_draft(history, stride, lengths, B, n, k, pad, drafts, count,
                                              static_cast<cudaStream_t>(stream)));
}

sv_status spec_verify_row_stats(const void *logits, int64_t batch_stride, int64_t row_stride,
                                sv_dtype dtype, int B, int rows_per_seq, int V,
                                float temperature, float *m_out, float *lse_out,
                                void *workspace, size_t workspace_bytes, void *stream) {
    if (!dtype_ok(dtype)) return SV_ERR_UNSUPPORTED;
    if (B < 0 || rows_per_seq < 1 || V < 1 || V > SV_MAX_VOCAB || batch_stride < 0 || row_stride < 0)
        return SV_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!logits || !m_out || !lse_out) return SV_ERR_INVALID_ARG;
    const int ntile = ntile_of(V, dtype);
    if (!tiles_fit(B, rows_per_seq, ntile) || int64_t(B) * rows_per_seq > kMaxGrid)
        return SV_ERR_INVALID_ARG;
    const Layout L = layout(SV_MODE_ROW_STATS, B, rows_per_seq, V, dtype);
    if (sv_status st = check_workspace(L, workspace, workspace_bytes)) return st;
    const bool vec = vec_ok(logits, batch_stride, row_stride, dtype);
    const Logits a{logits, batch_stride, row_stride};
    const float c = float(1.4426950408889634 / double(temperature));
    const float inv_t = float(1.0 / double(temperature));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *partial = at(workspace, L.partial);
    cudaError_t e = sv::launch_stats_tiles(dtype == SV_BF16, vec, a, rows_per_seq, a, rows_per_seq, B, V,
                                           ntile, c, partial, s);
    if (e == cudaSuccess)
        e = sv::launch_rowstats_finalize(B * rows_per_seq, ntile, c, inv_t, partial, m_out, lse_out, s);
    return cuda_status(e);
}

size_t spec_verify_status_offset(sv_mode mode, int B, int rows, int V, sv_dtype dtype) {
    if ((mode != SV_MODE_SAMPLE && mode != SV_MODE_TREE_SAMPLE && mode != SV_MODE_SAMPLE_LAZY &&
         mode != SV_MODE_TYPICAL && mode != SV_MODE_SAMPLE_ONEHOT) ||
        B <= 0 || rows < 0 || V <= 0 || !dtype_ok(dtype))
        return size_t(-1);
    return layout(mode, B, rows, V, dtype).rctl;
}

sv_status spec_verify_wait_selftest(int *ctl, int expected_arrivals, uint32_t limit_us, void *stream) {
    if (!ctl || expected_arrivals < 1 || expected_arrivals > 2 || limit_us > 5000000u) return SV_ERR_INVALID_ARG;
    return cuda_status(sv::launch_wait_selftest(ctl, expected_arrivals, uint64_t(limit_us) * 1000u,
                                                static_cast<cudaStream_t>(stream)));
}

sv_status spec_verify_exp_df(const float *y_hi, const float *y_lo, int n, float *out_hi, float *out_lo,
                             void *stream) {
    if (n < 0) return SV_ERR_INVALID_ARG;
    if (n == 0) return SV_OK;
    if (!y_hi || !y_lo || !out_hi || !out_lo) return SV_ERR_INVALID_ARG;
    return cuda_status(sv::launch_exp_df(y_hi, y_lo, n, out_hi, out_lo, static_cast<cudaStream_t>(stream)));
}

sv_status spec_verify_set_stage_events(void *const *events, int n_events) {
    if (n_events < 0 || n_events > kMaxStageEvents) return SV_ERR_INVALID_ARG;
    if (events == nullptr || n_events == 0) {
        t_nevents = 0;
        return SV_OK;
    }
    for (int i = 0; i < n_events; ++i) t_events[i] = static_cast<cudaEvent_t>(events[i]);
    t_nevents = n_events;
    return SV_OK;
}

sv_status spec_verify_uniforms(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                               float *out, void *stream) {
    if (B < 0 || positions < 0 || purpose < 0 || purpose > 1) return SV_ERR_INVALID_ARG;
    if (int64_t(B) * positions > kMaxGrid) return SV_ERR_INVALID_ARG;
    if (B == 0 || positions == 0) return SV_OK;
    if (!out) return SV_ERR_INVALID_ARG;
    return cuda_status(sv::launch_uniforms(seed, offset, B, positions, purpose, out,
                                           static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
