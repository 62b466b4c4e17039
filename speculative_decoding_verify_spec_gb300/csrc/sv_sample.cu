// sv_sample.cu -- the sampling path of the verifier.
//
// Method ("7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead": "The rule",
// "Extending to a chain of gamma draft tokens", apply_temperature / speculative_step of "A
// From-Scratch Implementation"; "Speculative Decoding: Draft Models, EAGLE, and How to
// Actually Use It": "The Algorithm"):
//   p_i = softmax(target_i / T), q_i = softmax(draft_i / T);
//   accept draft x_i with probability min(1, p_i(x_i) / q_i(x_i)), left to right;
//   at the first rejection k, draw the token from (p_k - q_k)+ normalised, and stop;
//   if all gamma drafts are accepted, draw a bonus token from p_gamma.
//
// GPU decomposition (one pass over every logit, then O(1) rows per sequence):
//   stats_tiles     persistent: every 4 KB tile of the 2 gamma + 1 rows of every sequence
//                   gives a NaN-propagating max M and sum 2^((l - M) log2(e) / T), one warp
//                   per tile.
//   decide          one warp per sequence: merge the tile partials into (M, S) per row,
//                   gather p_i(x_i), q_i(x_i), draw the Philox uniforms and scan.
//   residual_tiles  persistent: (sequences that rejected) the residual mass of every 2 KB
//                   residual tile of row k, one warp per tile.
//   draw            one warp per sequence: prefix over the unit masses (residual tiles, or
//                   the tiles of p for a bonus draw), then an in-order scan inside the chosen
//                   unit held in registers; the first j with C_j > u' R.
#include <algorithm>

#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_internal.h"
#include "sv_refine.cuh"

namespace sv {
namespace {

// Unnormalised target weight 2^((t - M) c) = exp((t - M) / T) with a single rounding of
// the (exact) difference times c.
__device__ __forceinline__ float weight(float x, float M, float c) {
    return ex2(__fmul_rn(__fsub_rn(x, M), c));
}

// (p_j - q_j)+ with p_j = 2^((t_j - M_t) c) / S_t and q_j likewise.  Both the tile-mass
// kernel and the in-unit scan call this one function, so the two agree bit for bit.  The
// products and the difference are explicitly rounded (no FMA contraction), so rows that
// are identical give exactly p_j - q_j = 0, as in exact arithmetic.
__device__ __forceinline__ float residual_weight(float tj, float dj, float c, float mt, float inv_st,
                                                 float md, float inv_sd) {
    const float p = __fmul_rn(weight(tj, mt, c), inv_st);
    const float q = __fmul_rn(weight(dj, md, c), inv_sd);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// residual_weight on two elements: the exponent arguments and the two products with FP32x2
// instructions, the difference p - q with one scalar subtraction per element.  A packed
// p + (-q) is not safe: the code generator may fuse the product q into that addition
// (one FFMA2, which keeps p's rounding error, so identical rows would leave ~1e-8 of
// residual mass instead of exactly 0), and scalar arithmetic with explicit rounding is
// never fused.  Each result equals residual_weight bit for bit.
__device__ __forceinline__ float2 residual_weight2(float2 t2, float2 d2, float2 c2, float2 nmt2, float2 inv_st2,
                                                   float2 nmd2, float2 inv_sd2) {
    const float2 yt = __fmul2_rn(__fadd2_rn(t2, nmt2), c2);
    const float2 yd = __fmul2_rn(__fadd2_rn(d2, nmd2), c2);
    const float2 p = __fmul2_rn(make_float2(ex2(yt.x), ex2(yt.y)), inv_st2);
    const float2 q = __fmul2_rn(make_float2(ex2(yd.x), ex2(yd.y)), inv_sd2);
    return make_float2(fmaxf(__fsub_rn(p.x, q.x), 0.f), fmaxf(__fsub_rn(p.y, q.y), 0.f));
}

// ------------------------------------------------------------------------------------
// Row statistics: partial[(seq * R + row) * ntile + tile] = (M, S) of that 4 KB tile, S
// relative to the tile's own maximum.  Local rows [0, rows_a) come from a, the rest from bt.
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 4)
    stats_tiles_kernel(Logits a, int rows_a, Logits bt, int R, int V, int ntile, int64_t items, float c,
                       float2 *__restrict__ partial) {
    griddep_launch_next();
    griddep_wait();  // before any read: the caller's previous kernel may be writing the logits
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * kWarps;
    for (TileWalk w(int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5), nwarps, R, ntile); w.it < items;
         w.next(nwarps)) {
        const char *rp = w.local < rows_a ? row_ptr(a, D::kBytes, w.seq, w.local)
                                          : row_ptr(bt, D::kBytes, w.seq, w.local - rows_a);
        const int64_t c0 = int64_t(w.tile) * tile_elems<D>();
        const int len = unit_len(V, c0, tile_elems<D>());
        uint4 v[kTileVecs];
#pragma unroll
        for (int u = 0; u < kTileVecs; ++u) {
            const int e0 = (lane + 32 * u) * D::EPV;
            v[u] = e0 < len ? load_vec<D, VEC>(rp, c0, e0, len) : neg_inf_vec<D>();
        }
        // the tile's maximum first (NaN-propagating); every lane then sums relative to it
        const float M = warp_reduce(thread_max<D>(v), [](float x, float y) { return max_nan(x, y); });
        float S = 0.f;
        if (is_finite(M)) S = warp_reduce(thread_sumexp<D>(v, c, M), [](float x, float y) { return x + y; });
        if (lane == 0 && SV_IN(w.it, items)) partial[w.it] = make_float2(M, S);
    }
}

// ------------------------------------------------------------------------------------
// Decide, one CTA per sequence: warp w merges the tile partials of rows w, w + kDecideWarps,
// ... into (M, S); warp 0 then runs the accept scan.
constexpr int kDecideWarps = 16;

// The decision of sequence seq by the NW warps of a CTA (after the previous kernel's data is
// visible): warp w merges the tile partials of rows w, w + NW, ... into (M, S) (s_stat:
// [2 gamma + 1]); warp 0 then runs the accept scan.  x0, tx0, dx0: lane i's (< gamma) draft
// token and its two logits, loaded by the caller.
template <class D, int NW>
__device__ __forceinline__ void decide_sequence(Logits t, Logits d, int B, int gamma, int V, int ntile, float c,
                                                const int32_t *__restrict__ x, uint64_t seed, uint64_t offset,
                                                const float2 *__restrict__ partial, float2 *__restrict__ rowstat,
                                                int2 *__restrict__ plan, int32_t *__restrict__ accepted_len,
                                                int32_t *__restrict__ out_tokens, int *__restrict__ rflag,
                                                int64_t seq, int32_t x0, float tx0, float dx0, float2 *s_stat) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = 2 * gamma + 1;
    for (int r = warp; r < R; r += NW) {
        const bool in = SV_IN((seq * R + r + 1) * ntile - 1, int64_t(B) * R * ntile);
        const float2 st = in ? warp_merge_stats(partial + (seq * R + r) * ntile, ntile, c, lane) : make_float2(0.f, 1.f);
        if (lane == 0) {
            s_stat[r] = st;
            if (SV_IN(seq * R + r, int64_t(B) * R)) rowstat[seq * R + r] = st;
        }
    }
    __syncthreads();
    if (warp != 0) return;

    bool ok = true;
    for (int r = lane; r < R; r += 32) ok &= is_finite(s_stat[r].x);
    for (int i = lane; i < gamma; i += 32) {
        const int32_t xi = i == lane ? x0 : x[seq * gamma + i];
        ok &= xi >= 0 && xi < V;
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    int32_t *out = out_tokens + seq * (gamma + 1);
    if (!SV_IN(seq, B)) return;
    if (!ok) {
        for (int i = lane; i <= gamma; i += 32) out[i] = -1;
        if (lane == 0) {
            accepted_len[seq] = -1;
            plan[seq] = make_int2(-1, -1);
            rflag[seq] = 0;
        }
        return;
    }

    // the scan; an accept test whose two sides u q and p are within the fp32 error of
    // each other marks the sequence for the extended-precision re-draw
    int k = gamma;
    bool near_any = false;
    for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        bool reject = false, near = false;
        if (i < gamma) {
            const float2 st = s_stat[i];
            const float2 sd = s_stat[gamma + 1 + i];
            float tx = tx0, dx = dx0;
            if (i0 > 0) {
                const int32_t xi = x[seq * gamma + i];
                tx = load_elem<D>(row_ptr(t, D::kBytes, seq, i), xi);
                dx = load_elem<D>(row_ptr(d, D::kBytes, seq, i), xi);
            }
            const float p = weight(tx, st.x, c) / st.y;
            const float q = weight(dx, sd.x, c) / sd.y;
            const float u = uniform01(seed, offset, uint32_t(seq), uint32_t(i), 0u);
            reject = !(u * q < p);
            near = fabsf(u * q - p) < kRefineAcceptWindow * fmaxf(p, u * q);
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, reject);
        const unsigned performed = m ? ((2u << (__ffs(m) - 1)) - 1u) : 0xFFFFFFFFu;  // up to the first rejection
        near_any |= (__ballot_sync(0xFFFFFFFFu, near) & performed) != 0u;
        if (m) {
            k = i0 + __ffs(m) - 1;
            break;
        }
    }
    for (int i = lane; i <= gamma; i += 32) {
        if (i < k) out[i] = x[seq * gamma + i];
        else if (i > k) out[i] = -1;
    }
    if (lane == 0) {
        accepted_len[seq] = k;
        plan[seq] = make_int2(k, k < gamma ? 1 : 0);
        rflag[seq] = near_any ? kRefineAccept : 0;
    }
}

template <class D>
__global__ void __launch_bounds__(kDecideWarps * 32)
    decide_kernel(Logits t, Logits d, int B, int gamma, int V, int ntile, float c,
                  const int32_t *__restrict__ x, uint64_t seed, uint64_t offset,
                  const float2 *__restrict__ partial, float2 *__restrict__ rowstat,
                  int2 *__restrict__ plan, int32_t *__restrict__ accepted_len,
                  int32_t *__restrict__ out_tokens, int *__restrict__ rflag, int *__restrict__ rctl,
                  int *__restrict__ rbar) {
    extern __shared__ float2 s_stat[];  // [2 gamma + 1]
    griddep_launch_next();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t seq = blockIdx.x;

    // the accept test's operands for the first 32 drafts do not depend on the statistics
    // (nor on an earlier kernel): their loads go out before the wait
    int32_t x0 = 0;
    float tx0 = 0.f, dx0 = 0.f;
    if (warp == 0 && lane < gamma) {
        x0 = x[seq * gamma + lane];
        if (x0 >= 0 && x0 < V) {
            tx0 = load_elem<D>(row_ptr(t, D::kBytes, seq, lane), x0);
            dx0 = load_elem<D>(row_ptr(d, D::kBytes, seq, lane), x0);
        }
    }
    griddep_wait();
    if (blockIdx.x == 0 && threadIdx.x < kRefineCtlWords) {  // this call's re-draw lists and barrier
        rctl[threadIdx.x] = 0;
        rbar[threadIdx.x] = 0;
    }
    decide_sequence<D, kDecideWarps>(t, d, B, gamma, V, ntile, c, x, seed, offset, partial, rowstat, plan,
                                     accepted_len, out_tokens, rflag, seq, x0, tx0, dx0, s_stat);
}

// ------------------------------------------------------------------------------------
// Residual masses: csum[seq * nrt + tile] = sum over the residual tile of (p - q)+ at the
// stop row, for the sequences that rejected (plan mode 1); other entries are not written.
// Persistent, with blocked work: warp w takes the items [w * per, (w + 1) * per), i.e.
// runs of consecutive tiles of one or two sequences, so a sequence's plan and statistics
// are read once per run and the warp's loads walk along the row.  The weights of element
// pairs come from residual_weight2 (FP32x2), even and odd elements summed separately.
// (Staging the tiles through shared memory with asynchronous copies made this kernel ~2 us
// faster but the re-draw kernel that follows it ~10 us slower; measured, not kept.)
constexpr bool kResidualPrefetch = false;  // load tile i + 1 of a run while computing tile i (measured: no gain)
constexpr int kResidualCtas = 4;           // resident CTAs per SM the kernel is built for

template <class D, bool VEC>
__device__ __forceinline__ void load_residual_tile(const char *tp, const char *dp, int64_t c0, int len, int lane,
                                                   uint4 (&tv)[kResVecs], uint4 (&dv)[kResVecs]) {
#pragma unroll
    for (int u = 0; u < kResVecs; ++u) {
        const int e0 = (lane + 32 * u) * D::EPV;
        tv[u] = e0 < len ? load_vec<D, VEC>(tp, c0, e0, len) : neg_inf_vec<D>();
        dv[u] = e0 < len ? load_vec<D, VEC>(dp, c0, e0, len) : neg_inf_vec<D>();
    }
}

// The residual mass sum (p - q)+ of one loaded residual tile (every lane returns it): element
// pairs in FP32x2, even and odd elements summed separately, then the warp.
template <class D>
__device__ __forceinline__ float residual_tile_mass(const uint4 (&tv)[kResVecs], const uint4 (&dv)[kResVecs], float c,
                                                    float2 st, float inv_st, float2 sd, float inv_sd) {
    float2 acc = make_float2(0.f, 0.f);
    const float2 c2 = make_float2(c, c), nmt2 = make_float2(-st.x, -st.x), inv_st2 = make_float2(inv_st, inv_st),
                 nmd2 = make_float2(-sd.x, -sd.x), inv_sd2 = make_float2(inv_sd, inv_sd);
#pragma unroll
    for (int u = 0; u < kResVecs; ++u) {
        const uint32_t tw[4] = {tv[u].x, tv[u].y, tv[u].z, tv[u].w}, dw[4] = {dv[u].x, dv[u].y, dv[u].z, dv[u].w};
#pragma unroll
        for (int q = 0; q < 4; q += (D::EPV == 8 ? 1 : 2)) {
            float2 t2, d2;
            if constexpr (D::EPV == 8) {
                t2 = make_float2(bf16_lo(tw[q]), bf16_hi(tw[q]));
                d2 = make_float2(bf16_lo(dw[q]), bf16_hi(dw[q]));
            } else {
                t2 = make_float2(__uint_as_float(tw[q]), __uint_as_float(tw[q + 1]));
                d2 = make_float2(__uint_as_float(dw[q]), __uint_as_float(dw[q + 1]));
            }
            acc = __fadd2_rn(acc, residual_weight2(t2, d2, c2, nmt2, inv_st2, nmd2, inv_sd2));
        }
    }
    return warp_reduce(acc.x + acc.y, [](float x, float y) { return x + y; });
}

template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, kResidualCtas)
    residual_tiles_kernel(Logits t, Logits d, int gamma, int V, int nrt, int64_t items, int64_t per, float c,
                          const float2 *__restrict__ rowstat, const int2 *__restrict__ plan,
                          float *__restrict__ csum) {
    griddep_wait();
    griddep_launch_next();  // after the wait: the draw's prologue may read what decide wrote
    const int lane = threadIdx.x & 31;
    const int R = 2 * gamma + 1;
    int64_t it = (int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * per;
    const int64_t end = it + per < items ? it + per : items;
    while (it < end) {
        const int64_t seq = it / nrt;
        const int64_t run_end = (seq + 1) * nrt < end ? (seq + 1) * nrt : end;
        const int2 pl = SV_IN(seq, items / nrt) ? plan[seq] : make_int2(-1, -1);
        if (pl.y == 1 && pl.x >= 0 && pl.x < gamma) {  // uniform over the warp (a plan out of range: no work)
            const int k = pl.x;
            const float2 st = rowstat[seq * R + k], sd = rowstat[seq * R + gamma + 1 + k];
            const float inv_st = 1.f / st.y, inv_sd = 1.f / sd.y;
            const char *tp = row_ptr(t, D::kBytes, seq, k);
            const char *dp = row_ptr(d, D::kBytes, seq, k);
            constexpr int RE = res_tile_elems<D>();
            uint4 tv[kResVecs], dv[kResVecs];
            load_residual_tile<D, VEC>(tp, dp, (it - seq * nrt) * RE, unit_len(V, (it - seq * nrt) * RE, RE), lane, tv,
                                       dv);
            for (; it < run_end; ++it) {
                uint4 ntv[kResVecs], ndv[kResVecs];
                if (kResidualPrefetch && it + 1 < run_end) {
                    const int64_t n0 = (it + 1 - seq * nrt) * RE;
                    load_residual_tile<D, VEC>(tp, dp, n0, unit_len(V, n0, RE), lane, ntv, ndv);
                }
                const float mass = residual_tile_mass<D>(tv, dv, c, st, inv_st, sd, inv_sd);
                if (lane == 0 && SV_IN(it, items)) csum[it] = mass;
                if (it + 1 < run_end) {
                    if (kResidualPrefetch) {
#pragma unroll
                        for (int u = 0; u < kResVecs; ++u) {
                            tv[u] = ntv[u];
                            dv[u] = ndv[u];
                        }
                    } else {
                        const int64_t n0 = (it + 1 - seq * nrt) * RE;
                        load_residual_tile<D, VEC>(tp, dp, n0, unit_len(V, n0, RE), lane, tv, dv);
                    }
                }
            }
        }
        it = run_end;
    }
}

// ------------------------------------------------------------------------------------
// The inverse-CDF draw of one sequence by one warp.  Units: mode 1 the residual tiles of the
// stop row (masses from residual_tiles), mode 0 the tiles of p (mass S_u 2^((M_u - M) c)
// from the row-statistics partials).  A zero residual falls back to p.  Lane l owns the
// contiguous units [l * per_lane, (l + 1) * per_lane); inside the chosen unit lane l holds
// a contiguous run of its vectors in registers, summed once and scanned once with the same
// arithmetic, so both passes see the same bits.  pl, st, sdk, flag0, u1: what decide wrote
// for the sequence (plan, statistics of its stop rows, its mark) and the draw's uniform.
template <class D, bool VEC>
__device__ __forceinline__ void draw_sequence(Logits t, Logits d, int B, int gamma, int V, int ntile, int nrt,
                                              int R, const int32_t *__restrict__ x, float c,
                                              const float2 *__restrict__ partial,
                                              const float *__restrict__ csum, int32_t *__restrict__ out_tokens,
                                              int *__restrict__ rflag, int *__restrict__ rctl,
                                              RefineInfo *__restrict__ rinfo, int64_t seq, int2 pl, float2 st,
                                              float2 sdk, int flag0, float u1,
                                              int lane) {
    if (pl.y < 0) return;  // invalid sequence: outputs already written by decide
    const int k = pl.x;
    int mode = pl.y == 1 ? 1 : 0;  // 1: residual after a rejection, 0: a draw from p
    // pl.y == 2 (a one-hot q rejected x_k): the draw from p without x_k, i.e. its tile's mass
    // less x_k's weight and x_k's own weight 0
    int ex = pl.y == 2 && SV_IN(seq * gamma + k, int64_t(B) * gamma) ? x[seq * gamma + k] : -1;
    if (ex >= 0 && !SV_IN(ex, V)) ex = -1;
    const float w_ex = ex >= 0 ? weight(load_elem<D>(row_ptr(t, D::kBytes, seq, k), ex), st.x, c) : 0.f;
    const int ex_tile = ex >= 0 ? ex / tile_elems<D>() : -1;
    const float2 *prow = partial + (seq * R + k) * ntile;
    const float *crow = csum + seq * nrt;
    auto unit_mass = [&](int u) -> float {
        if (mode) return SV_IN(seq * nrt + u, int64_t(B) * nrt) ? crow[u] : 0.f;
        if (!SV_IN((seq * R + k) * ntile + u, int64_t(B) * R * ntile)) return 0.f;
        const float2 p = prow[u];
        const float m = p.y * weight(p.x, st.x, c);  // mass of tile u under 2^((l - M) c)
        return u == ex_tile ? fmaxf(__fsub_rn(m, w_ex), 0.f) : m;
    };

    // this lane's first kKeep unit masses stay in registers for the walk below.  The prefixes
    // and the threshold are double-float (pair sums of the fp32 masses): the comparison is
    // then limited by the weights' own rounding, not by an fp32 running sum's resolution.
    constexpr int kKeep = 8;
    float keep[kKeep];
    df totd = df{0.f, 0.f}, incl = df{0.f, 0.f};
    int units = 0, per_lane = 0;
    for (int pass = 0; pass < 2; ++pass) {
        units = mode ? nrt : ntile;
        per_lane = (units + 31) / 32;
        PairSum lacc;
#pragma unroll
        for (int q = 0; q < kKeep; ++q) {
            const int u = lane * per_lane + q;
            keep[q] = (q < per_lane && u < units) ? unit_mass(u) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kKeep; ++q) lacc.add(keep[q]);
        for (int q = kKeep; q < per_lane; ++q) {
            const int u = lane * per_lane + q;
            if (u < units) lacc.add(unit_mass(u));
        }
        incl = df_warp_scan(lacc.value(), lane);
        totd = df_shfl(incl, 31);
        if ((mode == 1 || ex >= 0) && !(totd.hi > 0.f)) {  // exact-zero residual: draw from p
            mode = 0;
            ex = -1;
        } else {
            break;
        }
    }
    const df thr = df_mul_f(totd, u1);

    // the unit holding the threshold: the first lane whose range crosses it, then inside it
    int unit = -1;
    df base = df{0.f, 0.f};
    bool force_last = false, unit_fallback = false;
    const unsigned crossing = __ballot_sync(0xFFFFFFFFu, df_gt(incl, thr));
    if (crossing) {
        const int l = __ffs(crossing) - 1;
        df excl = df_shfl_up(incl, 1);
        if (lane == 0) excl = df{0.f, 0.f};
        if (lane == l) {
            df run = excl;
            int last_in_lane = lane * per_lane;
#pragma unroll
            for (int q = 0; q < kKeep; ++q) {
                const int u = lane * per_lane + q;
                if (unit < 0 && q < per_lane && u < units) {
                    last_in_lane = u;
                    const df nx = df_add(run, df_from(keep[q]));
                    if (df_gt(nx, thr)) unit = u;
                    else run = nx;
                }
            }
            for (int q = kKeep; q < per_lane && unit < 0; ++q) {
                const int u = lane * per_lane + q;
                if (u >= units) break;
                last_in_lane = u;
                const df nx = df_add(run, df_from(unit_mass(u)));
                if (df_gt(nx, thr)) unit = u;
                else run = nx;
            }
            if (unit < 0) {
                unit = last_in_lane;  // rounding: stay inside this lane's units
                unit_fallback = true;
            }
            base = run;
        }
        unit = __shfl_sync(0xFFFFFFFFu, unit, l);
        base = df_shfl(base, l);
        unit_fallback = __shfl_sync(0xFFFFFFFFu, unit_fallback, l);
    } else {  // rounding left the threshold at or above the total: the last unit with mass
        int lp = -1;
        for (int q = 0; q < per_lane; ++q) {
            const int u = lane * per_lane + q;
            if (u < units && unit_mass(u) > 0.f) lp = u;
        }
        lp = warp_reduce(lp, [](int a, int b) { return max(a, b); });
        unit = lp >= 0 ? lp : 0;
        force_last = true;
    }

    // inside the unit: lane l owns the contiguous vectors [l * VPL, (l + 1) * VPL)
    const int unit_elems = mode ? res_tile_elems<D>() : tile_elems<D>();
    const int last_unit = (V - 1) / unit_elems;  // units past it hold no element of the row
    if (unit > last_unit) unit = last_unit;
    const int VPL = mode ? kResVecs : kTileVecs;
    const float2 sd = mode ? sdk : make_float2(0.f, 1.f);
    const float inv_st = 1.f / st.y, inv_sd = 1.f / sd.y;
    const char *tp = row_ptr(t, D::kBytes, seq, k);
    const char *dp = row_ptr(d, D::kBytes, seq, k);
    const int64_t u0 = int64_t(unit) * unit_elems;
    const int len = unit_len(V, u0, unit_elems);
    uint4 tv[kTileVecs], dv[kResVecs];
#pragma unroll
    for (int v = 0; v < kTileVecs; ++v) {
        const int e0 = (lane * VPL + v) * D::EPV;
        tv[v] = (v < VPL && e0 < len) ? load_vec<D, VEC>(tp, u0, e0, len) : neg_inf_vec<D>();
    }
#pragma unroll
    for (int v = 0; v < kResVecs; ++v) {
        const int e0 = (lane * VPL + v) * D::EPV;
        dv[v] = (mode && e0 < len) ? load_vec<D, VEC>(dp, u0, e0, len) : neg_inf_vec<D>();
    }
    auto w_at = [&](const uint4 &t4, const uint4 &d4, int e, int j) -> float {  // j: index in the unit
        const float tj = vec_elem<D>(t4, e);
        return mode ? residual_weight(tj, vec_elem<D>(d4, e), c, st.x, inv_st, sd.x, inv_sd)
                    : (u0 + j == ex ? 0.f : weight(tj, st.x, c));
    };
    PairSum lsum;
    int lastpos = -1;
#pragma unroll
    for (int v = 0; v < kTileVecs; ++v) {
        if (v < VPL) {
            const int e0 = (lane * VPL + v) * D::EPV;
#pragma unroll
            for (int e = 0; e < D::EPV; ++e) {
                const float w = w_at(tv[v], dv[v % kResVecs], e, e0 + e);
                lsum.add(w);
                if (e0 + e < len && w > 0.f) lastpos = e0 + e;
            }
        }
    }
    const df lincl = df_warp_scan(lsum.value(), lane);
    df lexcl = df_shfl_up(lincl, 1);
    if (lane == 0) lexcl = df{0.f, 0.f};
    // the lane whose run crosses thr, then its logits spread over the warp (one or two per
    // lane, the same arithmetic from the same bits) and a second scan
    int first = kNoIndex;
    float g = 0.f;  // distance from thr to the nearer of C_{j-1} and C_j of the drawn j
    const unsigned lb = force_last ? 0u : __ballot_sync(0xFFFFFFFFu, df_gt(df_add(base, lincl), thr));
    if (lb) {
        const int l3 = __ffs(lb) - 1;
        const int NE = VPL * D::EPV;        // logits per lane of the unit
        const int ne2 = (NE + 31) / 32;     // ... per lane of this scan (1 or 2)
        const float inv_t1 = inv_st, inv_d1 = inv_sd;
        float w2[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int j = l3 * NE + lane * ne2 + r;
            if (r < ne2 && lane * ne2 + r < NE && j < len) {
                const float tj = load_elem<D>(tp, u0 + j);
                w2[r] = mode ? residual_weight(tj, load_elem<D>(dp, u0 + j), c, st.x, inv_t1, sd.x, inv_d1)
                             : (u0 + j == ex ? 0.f : weight(tj, st.x, c));
            }
        }
        PairSum ps;
        ps.add(w2[0]);
        ps.add(w2[1]);
        const df e_incl = df_warp_scan(ps.value(), lane);
        const df start = df_add(base, df_shfl(lexcl, l3));
        const unsigned eb = __ballot_sync(0xFFFFFFFFu, df_pos(df_sub(df_add(start, e_incl), thr)));
        if (eb) {
            const int l4 = __ffs(eb) - 1;
            df run2 = df_add(start, df_shfl(df_shfl_up(e_incl, 1), l4));
            if (l4 == 0) run2 = start;
            const float wa = __shfl_sync(0xFFFFFFFFu, w2[0], l4), wb = __shfl_sync(0xFFFFFFFFu, w2[1], l4);
            const df a0 = df_sub(df_add(run2, df_from(wa)), thr);  // C - thr after the first logit
            int r = 0;
            float w = wa;
            df above = a0;
            if (!df_pos(a0) && ne2 > 1) {
                r = 1;
                w = wb;
                above = df_sub(df_add(df_add(run2, df_from(wa)), df_from(wb)), thr);
            }
            if (df_pos(above)) {
                first = l3 * NE + l4 * ne2 + r;
                g = fminf(__fsub_rn(w, above.hi), above.hi);  // thr - C_{j-1} = w - (C_j - thr)
            }
        }
    }
    lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
    int tok = first != kNoIndex ? first : lastpos;
    if (tok < 0) tok = 0;
    // a draw whose threshold lies within the fp32 weights' error of a CDF boundary (or that
    // needed a rounding fallback, or a sequence decide marked) is redone in extended precision
    if (lane == 0) {
        if (SV_IN(seq * (gamma + 1) + k, int64_t(B) * (gamma + 1))) out_tokens[seq * (gamma + 1) + k] = int32_t(u0 + tok);
        const bool fell_back = (pl.y == 1 && mode == 0) || (pl.y == 2 && ex < 0);  // no residual mass
        // (a draw from p weighs in units of the row maximum's weight, not of S; without x_k its
        // tile's mass carries the subtraction's rounding too)
        const bool near = first == kNoIndex || force_last || unit_fallback || fell_back ||
                          !(g >= (mode ? kRefineCdfWindowRes * totd.hi + token_window(st.y) + token_window(sd.y)
                                       : kRefineCdfWindow * totd.hi + kTokenWindow * (fminf(1.f, st.y - 1.f) + w_ex)));
        int flag = flag0;
        if (near && flag == 0) flag = kRefineDraw;
        if (flag != 0) {  // listed: a marked accept test on the rescan list, a draw on the main list
            rflag[seq] = flag;
            atomicAdd(rctl + kRefineCount, 1);
            const int e = (flag & kRefineAccept) ? B + atomicAdd(rctl + kRefineAll, 1) : atomicAdd(rctl + kRefineMain, 1);
            if (SV_IN(e, 2 * int64_t(B))) rinfo[e] = RefineInfo{int(seq), flag, k, pl.y, st.x, st.y, sdk.x, sdk.y};
        }
    }
}

// ------------------------------------------------------------------------------------
// The draws and the re-draw in one cooperative grid (every CTA resident): each warp draws
// its sequences (grid-stride), then every CTA runs the re-draw's phases, which start with a
// grid barrier and end at once when no sequence was marked.  With `early` (the residual
// kernel ran in between and let this grid start only after its own wait on decide) a warp's
// first plan is read before the wait for the residual masses.
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
    draw_refine_kernel(Logits t, Logits d, int B, int gamma, int V, int ntile, int nrt, float c, float T,
                       uint64_t seed, uint64_t offset, int rule, int R, const int *__restrict__ lavail,
                       const int32_t *__restrict__ x, const float2 *__restrict__ partial,
                       const float2 *__restrict__ rowstat,
                       const int2 *__restrict__ plan, const float *__restrict__ csum,
                       int32_t *__restrict__ accepted_len, int32_t *__restrict__ out_tokens, int *__restrict__ rctl,
                       int *__restrict__ rbar, RefineInfo *__restrict__ rinfo, df *__restrict__ rsum,
                       int *__restrict__ ramb, df *__restrict__ rresc, bool early) {
    __shared__ RefineSmem sm;
    griddep_launch_next();
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nw = (int64_t(gridDim.x) * kThreads) >> 5;
    int *rflag = rctl + kRefineCtlWords;
    int2 pl = make_int2(-1, -1);
    float2 st = make_float2(0.f, 1.f), sdk = make_float2(0.f, 1.f);
    int flag0 = 0;
    float u1 = 0.f;
    auto read_plan = [&](int64_t seq) {
        pl = __ldcg(plan + seq);
        // a plan out of range (only if the kernel that writes plans stopped early) draws nothing
        if (pl.x < 0 || pl.x > gamma || pl.y < 0 || pl.y > 2 || (pl.y == 1 && pl.x == gamma)) pl = make_int2(-1, -1);
        st = make_float2(0.f, 1.f);
        sdk = make_float2(0.f, 1.f);
        flag0 = 0;
        if (pl.y >= 0 && SV_IN(seq * R + pl.x, int64_t(B) * R) &&
            (pl.y != 1 || SV_IN(seq * R + gamma + 1 + pl.x, int64_t(B) * R))) {
            st = __ldcg(rowstat + seq * R + pl.x);
            if (pl.y == 1) sdk = __ldcg(rowstat + seq * R + gamma + 1 + pl.x);
            flag0 = __ldcg(rflag + seq);
            u1 = uniform01(seed, offset, uint32_t(seq), uint32_t(pl.x), 1u);
        }
    };
    if (gw < B && early) read_plan(gw);
    griddep_wait();
    for (int64_t seq = gw; seq < B; seq += nw) {
        if (!(early && seq == gw)) read_plan(seq);
        if (pl.y >= 0)  // (an invalid sequence's outputs were written by decide)
            draw_sequence<D, VEC>(t, d, B, gamma, V, ntile, nrt, R, x, c, partial, csum, out_tokens, rflag, rctl,
                                  rinfo, seq, pl, st, sdk, flag0, u1, lane);
    }
    const RefineArgs ra{t, d, B, gamma, V, rule, R, lavail, T, seed, offset, x, rowstat, rctl, rbar, rinfo, rsum,
                        ramb, rresc, accepted_len, out_tokens};
    refine_phases<D>(ra, sm);
}

// ------------------------------------------------------------------------------------
// One sequence whose rows hold few tiles (B = 1, at most kSingleTiles tiles): the whole
// sampling call in ONE kernel of one CTA.  The stages are those of the four-kernel path --
// the rows' tile partials, decide_sequence, the residual masses of the stop row, the draw
// and the re-draw phases (a one-CTA grid meets at its grid barriers at once) -- each after
// a CTA barrier, with the same per-tile, per-sequence and re-draw code, so the outputs are
// the four-kernel path's bit for bit.  Such a call is bound by launch latency, not by its
// arithmetic; one launch replaces four.
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 1)
    single_sample_kernel(Logits t, Logits d, int gamma, int V, int ntile, int nrt, float c, float T, uint64_t seed,
                         uint64_t offset, const int32_t *__restrict__ x, float2 *__restrict__ partial,
                         float2 *__restrict__ rowstat, int2 *__restrict__ plan, float *__restrict__ csum,
                         int32_t *__restrict__ accepted_len, int32_t *__restrict__ out_tokens, int *__restrict__ rctl,
                         int *__restrict__ rbar, RefineInfo *__restrict__ rinfo, df *__restrict__ rsum,
                         int *__restrict__ ramb, df *__restrict__ rresc) {
    __shared__ RefineSmem sm;
    __shared__ float2 s_stat[kSingleTiles];
    griddep_launch_next();
    griddep_wait();  // before any read: the caller's previous kernel may be writing the inputs
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int R = 2 * gamma + 1;
    int *rflag = rctl + kRefineCtlWords;
    if (threadIdx.x < kRefineCtlWords) {  // this call's re-draw lists and barrier
        rctl[threadIdx.x] = 0;
        rbar[threadIdx.x] = 0;
    }
    // the rows' tile partials, a warp per tile
    const int items = R * ntile;
    for (int it = warp; it < items; it += kWarps) {
        const int local = it / ntile, tile = it - local * ntile;
        const char *rp = local <= gamma ? row_ptr(t, D::kBytes, 0, local) : row_ptr(d, D::kBytes, 0, local - gamma - 1);
        const int64_t c0 = int64_t(tile) * tile_elems<D>();
        const int len = unit_len(V, c0, tile_elems<D>());
        uint4 v[kTileVecs];
#pragma unroll
        for (int u = 0; u < kTileVecs; ++u) {
            const int e0 = (lane + 32 * u) * D::EPV;
            v[u] = e0 < len ? load_vec<D, VEC>(rp, c0, e0, len) : neg_inf_vec<D>();
        }
        const float M = warp_reduce(thread_max<D>(v), [](float a, float b) { return max_nan(a, b); });
        float S = 0.f;
        if (is_finite(M)) S = warp_reduce(thread_sumexp<D>(v, c, M), [](float a, float b) { return a + b; });
        if (lane == 0 && SV_IN(it, items)) partial[it] = make_float2(M, S);
    }
    int32_t x0 = 0;
    float tx0 = 0.f, dx0 = 0.f;
    if (warp == 0 && lane < gamma) {
        x0 = x[lane];
        if (x0 >= 0 && x0 < V) {
            tx0 = load_elem<D>(row_ptr(t, D::kBytes, 0, lane), x0);
            dx0 = load_elem<D>(row_ptr(d, D::kBytes, 0, lane), x0);
        }
    }
    __syncthreads();
    decide_sequence<D, kWarps>(t, d, 1, gamma, V, ntile, c, x, seed, offset, partial, rowstat, plan, accepted_len,
                               out_tokens, rflag, 0, x0, tx0, dx0, s_stat);
    __syncthreads();
    // the residual masses of the stop row, a warp per residual tile
    int2 pl = plan[0];
    if (pl.x < 0 || pl.x > gamma || pl.y < 0 || pl.y > 2 || (pl.y == 1 && pl.x == gamma)) pl = make_int2(-1, -1);
    if (pl.y == 1) {
        const int k = pl.x;
        const float2 st = rowstat[k], sd = rowstat[gamma + 1 + k];
        const float inv_st = 1.f / st.y, inv_sd = 1.f / sd.y;
        const char *tp = row_ptr(t, D::kBytes, 0, k), *dp = row_ptr(d, D::kBytes, 0, k);
        constexpr int RE = res_tile_elems<D>();
        for (int it = warp; it < nrt; it += kWarps) {
            uint4 tv[kResVecs], dv[kResVecs];
            load_residual_tile<D, VEC>(tp, dp, int64_t(it) * RE, unit_len(V, int64_t(it) * RE, RE), lane, tv, dv);
            const float mass = residual_tile_mass<D>(tv, dv, c, st, inv_st, sd, inv_sd);
            if (lane == 0 && SV_IN(it, nrt)) csum[it] = mass;
        }
    }
    __syncthreads();
    // the draw (warp 0), then the re-draw phases over the whole (one-CTA) grid
    if (warp == 0 && pl.y >= 0) {
        const float2 st = rowstat[pl.x];
        const float2 sdk = pl.y == 1 ? rowstat[gamma + 1 + pl.x] : make_float2(0.f, 1.f);
        const float u1 = uniform01(seed, offset, 0u, uint32_t(pl.x), 1u);
        draw_sequence<D, VEC>(t, d, 1, gamma, V, ntile, nrt, R, x, c, partial, csum, out_tokens, rflag, rctl, rinfo, 0,
                              pl, st, sdk, rflag[0], u1, lane);
    }
    __syncthreads();
    const RefineArgs ra{t, d, 1, gamma, V, kRuleSample, R, nullptr, T, seed, offset, x, rowstat, rctl, rbar, rinfo, rsum,
                        ramb, rresc, accepted_len, out_tokens};
    refine_phases<D>(ra, sm);
}

// ------------------------------------------------------------------------------------
__global__ void rowstats_finalize_kernel(int rows, int ntile, float c, float inv_t,
                                         const float2 *__restrict__ partial, float *__restrict__ m_out,
                                         float *__restrict__ lse_out) {
    griddep_launch_next();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // one warp per row
    if (r >= rows) return;
    const float2 s = warp_merge_stats(partial + r * ntile, ntile, c, lane);
    if (lane != 0) return;
    if (is_finite(s.x)) {
        const float m = s.x * inv_t;
        m_out[r] = m;
        lse_out[r] = m + logf(s.y);
    } else {
        m_out[r] = __int_as_float(0x7fc00000);
        lse_out[r] = __int_as_float(0x7fc00000);
    }
}

__global__ void uniforms_kernel(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                                float *__restrict__ out) {
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= int64_t(B) * positions) return;
    const int64_t b = idx / positions;
    const int i = int(idx - b * positions);
    out[idx] = uniform01(seed, offset, uint32_t(b), uint32_t(i), uint32_t(purpose));
}

}  // namespace

// ------------------------------------------------------------------------------------
// Launchers
// ------------------------------------------------------------------------------------
template <class KB1, class KB0, class KF1, class KF0>
inline auto pick(int dtype, bool vec, KB1 b1, KB0 b0, KF1 f1, KF0 f0) {
    return dtype == 1 ? (vec ? b1 : b0) : (vec ? f1 : f0);
}

cudaError_t launch_stats_tiles(int dtype, bool vec, Logits a, int rows_a, Logits b, int R, int B, int V,
                               int ntile, float c, void *partial, cudaStream_t s) {
    const int64_t items = int64_t(B) * R * ntile;
    auto k = pick(dtype, vec, stats_tiles_kernel<BF16, true>, stats_tiles_kernel<BF16, false>,
                  stats_tiles_kernel<F32, true>, stats_tiles_kernel<F32, false>);
    unsigned grid = 0;
    cudaError_t e = persistent_grid(k, items, &grid);
    if (e != cudaSuccess) return e;
    return launch_after(k, grid, kThreads, 0, s, a, rows_a, b, R, V, ntile, items, c, static_cast<float2 *>(partial));
}

cudaError_t launch_decide(int dtype, Logits t, Logits d, int B, int gamma, int V, int ntile,
                          float c, const int32_t *x, uint64_t seed, uint64_t offset,
                          const void *partial, void *rowstat, void *plan, int32_t *accepted_len,
                          int32_t *out_tokens, int *rflag, int *rctl, int *rbar, cudaStream_t s) {
    auto k = dtype == 1 ? decide_kernel<BF16> : decide_kernel<F32>;
    const size_t smem = size_t(2 * gamma + 1) * sizeof(float2);
    return launch_after(k, unsigned(B), kDecideWarps * 32, smem, s, t, d, B, gamma, V, ntile, c, x, seed, offset,
                        static_cast<const float2 *>(partial), static_cast<float2 *>(rowstat),
                        static_cast<int2 *>(plan), accepted_len, out_tokens, rflag, rctl, rbar);
}

cudaError_t launch_residual_tiles(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V,
                                  int nrt, float c, const void *rowstat, const void *plan, float *csum,
                                  cudaStream_t s) {
    const int64_t items = int64_t(B) * nrt;
    auto k = pick(dtype, vec, residual_tiles_kernel<BF16, true>, residual_tiles_kernel<BF16, false>,
                  residual_tiles_kernel<F32, true>, residual_tiles_kernel<F32, false>);
    unsigned grid = 0;
    cudaError_t e = persistent_grid(k, items, &grid);
    if (e != cudaSuccess) return e;
    const int64_t nwarps = int64_t(grid) * kWarps;
    const int64_t per = (items + nwarps - 1) / nwarps;
    return launch_after(k, grid, kThreads, 0, s, t, d, gamma, V, nrt, items, per, c,
                        static_cast<const float2 *>(rowstat), static_cast<const int2 *>(plan), csum);
}

bool single_sample_fits(int B, int gamma, int ntile) { return B == 1 && (2 * int64_t(gamma) + 1) * ntile <= kSingleTiles; }

cudaError_t launch_single_sample(int dtype, bool vec, Logits t, Logits d, int gamma, int V, int ntile, int nrt,
                                 float c, float T, uint64_t seed, uint64_t offset, const int32_t *x, void *partial,
                                 void *rowstat, void *plan, float *csum, int32_t *accepted_len, int32_t *out_tokens,
                                 int *rctl, int *rbar, RefineInfo *rinfo, void *rsum, int *ramb, void *rresc,
                                 cudaStream_t s) {
    auto k = pick(dtype, vec, single_sample_kernel<BF16, true>, single_sample_kernel<BF16, false>,
                  single_sample_kernel<F32, true>, single_sample_kernel<F32, false>);
    return launch_after(k, 1u, kThreads, 0, s, t, d, gamma, V, ntile, nrt, c, T, seed, offset, x,
                        static_cast<float2 *>(partial), static_cast<float2 *>(rowstat), static_cast<int2 *>(plan), csum,
                        accepted_len, out_tokens, rctl, rbar, rinfo, static_cast<df *>(rsum), ramb,
                        static_cast<df *>(rresc));
}

cudaError_t launch_draw_refine(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V, int ntile, int nrt,
                               float c, float T, uint64_t seed, uint64_t offset, int rule, int R, const int *lavail,
                               const int32_t *x, const void *partial,
                               const void *rowstat, const void *plan, const float *csum, int32_t *accepted_len,
                               int32_t *out_tokens, int *rctl, int *rbar, RefineInfo *rinfo, void *rsum, int *ramb,
                               void *rresc, bool early, cudaStream_t s) {
    auto k = pick(dtype, vec, draw_refine_kernel<BF16, true>, draw_refine_kernel<BF16, false>,
                  draw_refine_kernel<F32, true>, draw_refine_kernel<F32, false>);
    // every resident slot, or fewer for a small problem: a warp per sequence for the draws
    // and a warp per two units of a listed row pair for the re-draw's grid-wide phase (a
    // grid of one or two CTAs meets at its barriers at once)
    unsigned grid = 0;
    const int64_t warps = std::max<int64_t>(B, int64_t(B) * refine_units(V) / 2);
    cudaError_t e = persistent_grid(k, warps, &grid);
    if (e != cudaSuccess) return e;
    return launch_after_ex(true, k, grid, kThreads, 0, s, t, d, B, gamma, V, ntile, nrt, c, T, seed, offset, rule, R,
                           lavail, x,
                           static_cast<const float2 *>(partial), static_cast<const float2 *>(rowstat),
                           static_cast<const int2 *>(plan), csum, accepted_len, out_tokens, rctl, rbar, rinfo,
                           static_cast<df *>(rsum), ramb, static_cast<df *>(rresc), early);
}

cudaError_t launch_rowstats_finalize(int rows, int ntile, float c, float inv_t, const void *partial,
                                     float *m_out, float *lse_out, cudaStream_t s) {
    const unsigned grid = unsigned((int64_t(rows) * 32 + 255) / 256);
    return launch_after(rowstats_finalize_kernel, grid, 256, 0, s, rows, ntile, c, inv_t,
                        static_cast<const float2 *>(partial), m_out, lse_out);
}

cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                            float *out, cudaStream_t s) {
    const int64_t n = int64_t(B) * positions;
    const unsigned grid = unsigned((n + 255) / 256);
    uniforms_kernel<<<grid, 256, 0, s>>>(seed, offset, B, positions, purpose, out);
    return cudaGetLastError();
}

}  // namespace sv
