// sv_refine.cuh -- the extended-precision re-draw of near-boundary sampling sequences: the
// phases that the cooperative draw kernel (sv_sample.cu) runs after its draws.
//
// The sampler's decisions are comparisons of sums of exponentials: u q(x) < p(x) for an
// accept test, C_j > u' R for the inverse CDF (first page, "The rule"; R3 of the readings).
// In fp32 a comparison whose two sides differ by less than ~1e-7 relative can come out the
// other way than in exact arithmetic.  decide and draw mark such sequences (margins below
// their windows, which sit above the fp32 error) and list every one of them; these phases
// redo all of them in double-float arithmetic (sv_df.cuh, ~48 bits), which resolves every
// comparison whose exact margin is above ~1e-13.
//
// Lists: the main list (a draw to redo on a known stop row k: target and draft row k after
// a rejection, target row gamma for a bonus draw) and the rescan list (an accept test was
// near).  Units are 64 logits (two per lane of a warp).  Every phase ends at a grid barrier
// (the launch is cooperative, so every CTA is resident):
//   (the draws, then the barrier -- with nothing listed every CTA returns here)
//   R   rescan list, in chunks of kRescanChunk: every warp the unit sums of every row of the
//       chunk's sequences; then one CTA per sequence takes the row sums, runs the accept
//       tests again (u e_d(x) S_t < e_t(x) S_d), writes the accepted prefix, and either
//       draws the bonus token at once or appends the sequence to the main list at its new
//       stop row;
//   A   main list, every warp, one item per unit: the unit sums of exp((x - M) / T) of the
//       stop row (and of the draft row after a rejection), plus -- for a residual -- the same
//       sums over the logits where p > q for certain given the fp32 row sums (the sign of
//       p - q is that of e_t S_d - e_d S_t), and a count of the logits too near that ratio;
//   F   main list, one CTA per sequence: the exact row sums, rho = S_t / S_d; the residual's
//       unit masses pos_t - rho pos_d, plus, in a unit with near logits, their exact
//       max(e_t - rho e_d, 0); the unit holding u' x total by a block scan, the token inside
//       it by warp 0 (exact weights).  With no residual mass at all the draw comes from p on
//       that row (reading R4).
#pragma once

#include "spec_verify.h"
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_grid.cuh"
#include "sv_internal.h"

namespace sv {

struct RefineArgs {
    Logits t, d;
    int B, gamma, V;
    int rule;                   // kRuleSample, kRuleOnehot or kRuleTypical
    int R;                      // rows per sequence in rowstat: 2 gamma + 1 (chain), else gamma + 1
    const int *lavail;          // rows 0 .. lavail[b] - 1 read by a lazy walk (NULL: every row)
    float T;
    uint64_t seed, offset;
    const int32_t *x;           // draft tokens [B][gamma]
    const float2 *rowstat;      // (M, S) per row: target rows 0 .. gamma, then draft rows
    int *rctl;                  // control words (kRefine*), then the marks
    int *rbar;                  // the grid barrier's words (zeroed by decide)
    RefineInfo *rinfo;          // main list [0, B), rescan list [B, 2B)
    df *rsum;                   // main list: B x 5 x nu unit sums (all_t, all_d, pos_t, pos_d, fix)
    int *ramb;                  // main list: B x nu near-logit counts
    df *rresc;                  // rescan chunk: kRescanChunk x (2 gamma + 1) x nu unit sums
    int32_t *accepted_len, *out_tokens;
};

struct RefineSmem {
    df wsum[kWarps];
    df incl[kThreads];
    int i0, i1, unit;
    df base, total;
};

namespace refine {

constexpr int kLane = 2;             // logits per lane in a unit
constexpr int kUnit = 32 * kLane;    // 64 logits per unit (one warp)
constexpr float kSignBand = 4e-6f;   // relative band around S_t / S_d left to the exact pass
constexpr int kBatch = 8;            // values a thread loads together before it adds them

__device__ __forceinline__ df ldcg_df(const df *p) {
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(p));
    return df{v.x, v.y};
}
__device__ __forceinline__ void st_df(df *p, df v) { *reinterpret_cast<float2 *>(p) = make_float2(v.hi, v.lo); }
__device__ __forceinline__ df df_zero() { return df{0.f, 0.f}; }
// A record written by another SM earlier in this grid: read at L2.
__device__ __forceinline__ RefineInfo ldcg_info(const RefineInfo *p) {
    const int4 a = __ldcg(reinterpret_cast<const int4 *>(p)), b = __ldcg(reinterpret_cast<const int4 *>(p) + 1);
    return RefineInfo{a.x, a.y, a.z, a.w, __int_as_float(b.x), __int_as_float(b.y), __int_as_float(b.z),
                      __int_as_float(b.w)};
}

// exp((x_j - M) / T) of this lane's logits of unit u (0 past the row's end).  Every lane of
// the warp calls it together (the exponential's table comes by shuffle); tj = this lane's
// entry of that table.
template <class D>
__device__ __forceinline__ void lane_exps(const char *row, float M, df inv_t, int V, int u, int lane, float2 tj,
                                          df (&w)[kLane]) {
    const int64_t j0 = int64_t(u) * kUnit + lane * kLane;
    float xv[kLane];
#pragma unroll
    for (int e = 0; e < kLane; ++e) xv[e] = j0 + e < V ? load_elem<D>(row, j0 + e) : -__int_as_float(0x7f800000);
#pragma unroll
    for (int e = 0; e < kLane; ++e) w[e] = weight_df_warp(xv[e], M, inv_t, tj);
}

// lane_exps of one unit of two rows, all four loads issued before any exponential.
template <class D>
__device__ __forceinline__ void lane_exps2(const char *row_a, float Ma, const char *row_b, float Mb, df inv_t, int V,
                                           int u, int lane, float2 tj, df (&wa)[kLane], df (&wb)[kLane]) {
    const int64_t j0 = int64_t(u) * kUnit + lane * kLane;
    float xa[kLane], xb[kLane];
#pragma unroll
    for (int e = 0; e < kLane; ++e) {
        xa[e] = j0 + e < V ? load_elem<D>(row_a, j0 + e) : -__int_as_float(0x7f800000);
        xb[e] = j0 + e < V ? load_elem<D>(row_b, j0 + e) : -__int_as_float(0x7f800000);
    }
#pragma unroll
    for (int e = 0; e < kLane; ++e) {
        wa[e] = weight_df_warp(xa[e], Ma, inv_t, tj);
        wb[e] = weight_df_warp(xb[e], Mb, inv_t, tj);
    }
}

// The warp's sum of one value per lane, in lane order (every lane gets it).
__device__ __forceinline__ df warp_sum_ordered(df v, int lane) { return df_shfl(df_warp_scan(v, lane), 31); }

// Inclusive scan of one value per thread in thread order; every thread gets the block total.
__device__ __forceinline__ df block_scan(df v, RefineSmem &sm, df *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const df incl = df_warp_scan(v, lane);
    __syncthreads();
    if (lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    df before = df_zero(), all = df_zero();
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before = df_add(before, sm.wsum[w]);
        all = df_add(all, sm.wsum[w]);
    }
    *total = all;
    return df_add(before, incl);
}

// The inverse-CDF search at unit granularity over n unit masses val(i), by the whole CTA:
// thread t owns the contiguous run [t per, (t + 1) per).  *total = the sum of all of them
// (in this order); thr = *total x u.  Returns the first unit i with val(0) + ... + val(i) > thr
// and *base = the prefix before it; when rounding leaves no crossing (or the total is 0),
// the last unit with a positive mass and *force = true.  Every thread returns the same.
template <class Val>
__device__ __forceinline__ int block_search(int n, float u, Val val, df *total, df *thr, df *base, bool *force,
                                            RefineSmem &sm) {
    const int per = (n + kThreads - 1) / kThreads;
    df run = df_zero();
    int lp = -1;
    for (int q0 = 0; q0 < per; q0 += kBatch) {  // the loads of a batch all in flight together
        df v[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = int(threadIdx.x) * per + q0 + q;
            v[q] = (q0 + q < per && i < n) ? val(i) : df_zero();
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = int(threadIdx.x) * per + q0 + q;
            if (q0 + q < per && i < n) {
                run = df_add(run, v[q]);
                if (df_pos(v[q])) lp = i;
            }
        }
    }
    const df incl = block_scan(run, sm, total);
    *thr = df_mul_f(*total, u);
    sm.incl[threadIdx.x] = incl;
    if (threadIdx.x == 0) {
        sm.i0 = kThreads;
        sm.i1 = -1;
    }
    __syncthreads();
    if (df_gt(incl, *thr)) atomicMin(&sm.i0, int(threadIdx.x));
    if (lp >= 0) atomicMax(&sm.i1, lp);
    __syncthreads();
    const int first = sm.i0;
    if (int(threadIdx.x) == first) {  // walk this thread's run in the order it was summed
        df r = first > 0 ? sm.incl[first - 1] : df_zero();
        int unit = -1, last = first * per;
        for (int q0 = 0; q0 < per && unit < 0; q0 += kBatch) {  // a batch's loads in flight together
            df v[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int i = first * per + q0 + q;
                v[q] = (q0 + q < per && i < n) ? val(i) : df_zero();
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int i = first * per + q0 + q;
                if (unit < 0 && q0 + q < per && i < n) {
                    last = i;
                    const df nx = df_add(r, v[q]);
                    if (df_gt(nx, *thr)) unit = i;
                    else r = nx;
                }
            }
        }
        sm.unit = unit >= 0 ? unit : last;
        sm.base = r;
    }
    __syncthreads();
    int unit;
    if (first < kThreads) {
        unit = sm.unit;
        *base = sm.base;
        *force = false;
    } else {
        unit = sm.i1 >= 0 ? sm.i1 : 0;
        *base = df_zero();
        *force = true;
    }
    __syncthreads();
    return unit;
}

// The block sums of two lists of n values va(i), vb(i) in block_search's order.
template <class VA, class VB>
__device__ __forceinline__ void block_sum2(int n, VA va, VB vb, df *sa, df *sb, RefineSmem &sm) {
    const int per = (n + kThreads - 1) / kThreads;
    df ra = df_zero(), rb = df_zero();
    for (int q0 = 0; q0 < per; q0 += kBatch) {
        df a[kBatch], b[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = int(threadIdx.x) * per + q0 + q;
            const bool in = q0 + q < per && i < n;
            a[q] = in ? va(i) : df_zero();
            b[q] = in ? vb(i) : df_zero();
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            if (q0 + q < per && int(threadIdx.x) * per + q0 + q < n) {
                ra = df_add(ra, a[q]);
                rb = df_add(rb, b[q]);
            }
        }
    }
    block_scan(ra, sm, sa);
    block_scan(rb, sm, sb);
}

// Inside unit u (warp 0): the first logit whose prefix base + w(0) + ... + w(j) exceeds thr,
// with w this lane's kLane weights (index order); rounding past the unit's end, or force:
// the last logit with a positive weight (the unit's first logit if none).
__device__ __forceinline__ int unit_pick(const df (&w)[kLane], int u, int V, df base, df thr, bool force, int lane) {
    const int64_t j0 = int64_t(u) * kUnit + lane * kLane;
    df ls = df_zero();
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < kLane; ++e) {
        ls = df_add(ls, w[e]);
        if (j0 + e < V && df_pos(w[e])) lastpos = int(j0) + e;
    }
    lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
    int tok = lastpos;
    if (!force) {
        const df incl = df_warp_scan(ls, lane);
        df excl = df_shfl_up(incl, 1);
        if (lane == 0) excl = df_zero();
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, df_gt(df_add(base, incl), thr));
        if (bal) {
            const int l = __ffs(bal) - 1;
            int cand = -1, lpos = -1;
            df r2 = df_add(base, excl);
#pragma unroll
            for (int e = 0; e < kLane; ++e) {
                r2 = df_add(r2, w[e]);
                if (cand < 0 && j0 + e < V && df_gt(r2, thr)) cand = int(j0) + e;
                if (j0 + e < V && df_pos(w[e])) lpos = int(j0) + e;
            }
            if (cand < 0) cand = lpos;
            cand = __shfl_sync(0xFFFFFFFFu, cand, l);
            if (cand >= 0) tok = cand;
        }
    }
    return tok >= 0 ? tok : int(int64_t(u) * kUnit);
}

}  // namespace refine

// The phases after the draws (see the top of this file).  Every CTA of the cooperative grid
// calls this once, after its last draw.
template <class D>
__device__ void refine_phases(const RefineArgs &a, RefineSmem &sm) {
    using namespace refine;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto barrier = [&]() -> bool {
        if (grid_barrier(a.rbar)) return true;
        if (tid == 0) atomicExch(a.rctl + kRefineStatus, int(SV_ERR_TIMEOUT));
        return false;
    };
    if (!barrier()) return;  // every draw done, the lists complete
    const int nall = __ldcg(a.rctl + kRefineAll);
    if (__ldcg(a.rctl + kRefineMain) + nall == 0) return;  // (the same for every CTA)
    const int gamma = a.gamma, V = a.V, B = a.B, R = a.R;
    const bool onehot = a.rule == kRuleOnehot;
    const int nu = (V + kUnit - 1) / kUnit;
    const int64_t gw = (int64_t(blockIdx.x) * kThreads + tid) >> 5;
    const int64_t nw = (int64_t(gridDim.x) * kThreads) >> 5;
    const df inv_t = df_div(df_from(1.f), df_from(a.T));
    const float2 tj = kExp2Sixteenths[lane & 15];
    auto trow = [&](int64_t seq, int r) { return row_ptr(a.t, D::kBytes, seq, r); };
    auto drow = [&](int64_t seq, int r) { return row_ptr(a.d, D::kBytes, seq, r); };
    // rowstat index ri: target rows 0 .. gamma, then draft rows gamma + 1 .. 2 gamma
    auto stat_row = [&](int64_t seq, int ri) { return ri <= gamma ? trow(seq, ri) : drow(seq, ri - gamma - 1); };
    auto resid = [](df et, df ed, df rho) {  // max(e_t - rho e_d, 0): (p - q)+ in units of S_t
        const df w = df_sub(et, df_mul(rho, ed));
        return df_pos(w) ? w : df_zero();
    };
    // The token inside unit u (warp 0 computes; every thread returns it): the weights of
    // target row k, or with resid the residual weights of row pair k.
    auto pick = [&](int64_t seq, int k, float Mt, float Md, df rho, bool with_resid, int u, df b0, df thr,
                    bool force, int ex = -1) -> int {
        if (warp == 0) {
            df w[kLane];
            if (with_resid) {
                df wd[kLane];
                lane_exps2<D>(trow(seq, k), Mt, drow(seq, k), Md, inv_t, V, u, lane, tj, w, wd);
#pragma unroll
                for (int e = 0; e < kLane; ++e) w[e] = resid(w[e], wd[e], rho);
            } else {
                lane_exps<D>(trow(seq, k), Mt, inv_t, V, u, lane, tj, w);
#pragma unroll
                for (int e = 0; e < kLane; ++e)
                    if (int64_t(u) * kUnit + lane * kLane + e == ex) w[e] = df_zero();  // the excluded token
            }
            const int tok = unit_pick(w, u, V, b0, thr, force, lane);
            if (lane == 0) sm.unit = tok;
        }
        __syncthreads();
        const int tok = sm.unit;
        __syncthreads();
        return tok;
    };
    auto finish = [&](int64_t seq, int k, int tok) {  // thread 0
        if (SV_IN(seq * (gamma + 1) + k, int64_t(B) * (gamma + 1))) a.out_tokens[seq * (gamma + 1) + k] = int32_t(tok);
        atomicAdd(a.rctl + kRefineRedone, 1);
    };

    // R: the rescan list, kRescanChunk sequences at a time.
    for (int c0 = 0; c0 < nall; c0 += kRescanChunk) {
        const int nc = min(kRescanChunk, nall - c0);
        const int64_t items = int64_t(nc) * R * nu;
        for (int64_t it = gw; it < items; it += nw) {
            const int c = int(it / (int64_t(R) * nu));
            const int loc = int(it - int64_t(c) * R * nu);
            const int ri = loc / nu, u = loc - ri * nu;
            if (!SV_IN(B + c0 + c, 2 * int64_t(B))) continue;
            const int64_t seq = ldcg_info(a.rinfo + B + c0 + c).seq;
            if (!SV_IN(seq * R + ri, int64_t(B) * R) || !SV_IN((int64_t(c) * R + ri) * nu + u, int64_t(kRescanChunk) * R * nu))
                continue;
            const int avail = a.lavail ? __ldcg(a.lavail + seq) : gamma + 1;
            if ((ri <= gamma ? ri : ri - gamma - 1) >= avail) continue;  // a row the lazy walk did not read
            df w[kLane];
            lane_exps<D>(stat_row(seq, ri), a.rowstat[seq * R + ri].x, inv_t, V, u, lane, tj, w);
            const df s = warp_sum_ordered(df_add(w[0], w[1]), lane);
            if (lane == 0) st_df(a.rresc + (int64_t(c) * R + ri) * nu + u, s);
        }
        if (!barrier()) return;
        for (int c = blockIdx.x; c < nc; c += gridDim.x) {
            if (!SV_IN(B + c0 + c, 2 * int64_t(B))) continue;  // (uniform over the CTA)
            RefineInfo info = ldcg_info(a.rinfo + B + c0 + c);
            const int64_t seq = info.seq;
            if (!SV_IN(seq, B)) continue;
            const df *rs = a.rresc + int64_t(c) * R * nu;
            const int avail = a.lavail ? __ldcg(a.lavail + seq) : gamma + 1;
            int k2 = gamma;
            bool bad = false;  // the walk reaches a row the lazy walk could not read (not a distribution)
            for (int i = 0; i < gamma; ++i) {  // u e_d(x) S_t < e_t(x) S_d (one-hot: u S_t < e_t(x)), left to right
                if (i >= avail) {
                    bad = true;
                    break;
                }
                df St, Sd = df_from(1.f);
                block_sum2(nu, [&](int q) { return ldcg_df(rs + int64_t(i) * nu + q); },
                           [&](int q) { return onehot ? df_zero() : ldcg_df(rs + int64_t(gamma + 1 + i) * nu + q); },
                           &St, &Sd, sm);
                if (tid == 0) {
                    const int32_t xi = a.x[seq * gamma + i];
                    const df et = weight_df(load_elem<D>(trow(seq, i), xi), a.rowstat[seq * R + i].x, inv_t);
                    const float uu = uniform01(a.seed, a.offset, uint32_t(seq), uint32_t(i), 0u);
                    if (onehot) {
                        sm.i0 = df_lt(df_mul_f(St, uu), et) ? 0 : 1;
                    } else {
                        const df ed = weight_df(load_elem<D>(drow(seq, i), xi), a.rowstat[seq * R + gamma + 1 + i].x, inv_t);
                        sm.i0 = df_lt(df_mul_f(df_mul(ed, St), uu), df_mul(et, Sd)) ? 0 : 1;
                    }
                }
                __syncthreads();
                const int rejected = sm.i0;
                __syncthreads();
                if (rejected) {
                    k2 = i;
                    break;
                }
            }
            if (k2 == gamma && gamma >= avail) bad = true;
            int32_t *out = a.out_tokens + seq * (gamma + 1);
            for (int i = tid; i <= gamma; i += kThreads) {
                if (bad) out[i] = -1;
                else if (i < k2) out[i] = a.x[seq * gamma + i];
                else if (i > k2) out[i] = -1;
            }
            if (tid == 0) a.accepted_len[seq] = bad ? -1 : k2;
            if (bad) {
                if (tid == 0) atomicAdd(a.rctl + kRefineRedone, 1);
            } else if (k2 == gamma) {  // every draft accepted: the bonus draw from p_gamma, now
                df total, thr, b0;
                bool force;
                const int u = block_search(nu, uniform01(a.seed, a.offset, uint32_t(seq), uint32_t(gamma), 1u),
                                           [&](int q) { return ldcg_df(rs + int64_t(gamma) * nu + q); }, &total, &thr,
                                           &b0, &force, sm);
                const int tok = pick(seq, gamma, a.rowstat[seq * R + gamma].x, 0.f, df_zero(), false, u, b0, thr, force);
                if (tid == 0) finish(seq, gamma, tok);
            } else if (tid == 0) {  // a residual draw at the new stop row: onto the main list
                info.k = k2;
                info.mode = onehot ? 2 : 1;
                const int pos = atomicAdd(a.rctl + kRefineMain, 1);
                const float2 st2 = a.rowstat[seq * R + k2];
                const float2 sd2 = onehot ? make_float2(0.f, 1.f) : a.rowstat[seq * R + gamma + 1 + k2];
                info.Mt = st2.x;
                info.St = st2.y;
                info.Md = sd2.x;
                info.Sd = sd2.y;
                if (SV_IN(pos, B)) a.rinfo[pos] = info;
            }
            __syncthreads();
        }
        if (!barrier()) return;
    }

    // A: the main list, one item per unit.
    const int nmain = __ldcg(a.rctl + kRefineMain);
    const int64_t slot = int64_t(5) * nu;  // all_t, all_d, pos_t, pos_d, fix
    const int64_t na = int64_t(nmain) * nu;
    for (int64_t it = gw; it < na; it += nw) {
        const int e = int(it / nu), u = int(it - int64_t(e) * nu);
        if (!SV_IN(e, B)) continue;
        const RefineInfo info = ldcg_info(a.rinfo + e);
        const int64_t seq = info.seq;
        if (!SV_IN(seq, B) || !SV_IN(info.k, gamma + 1)) continue;
        const int k = info.k;
        df *S = a.rsum + e * slot;
        const float2 st = make_float2(info.Mt, info.St);  // the draw's copy of rowstat (no extra read)
        df wt[kLane];
        if (info.mode != 1) {  // a draw from p (a bonus draw, or p without a one-hot q's token): its sums only
            lane_exps<D>(trow(seq, k), st.x, inv_t, V, u, lane, tj, wt);
            const df at = warp_sum_ordered(df_add(wt[0], wt[1]), lane);
            if (lane == 0) st_df(S + u, at);
            continue;
        }
        const float2 sd = make_float2(info.Md, info.Sd);
        df wd[kLane];
        lane_exps2<D>(trow(seq, k), st.x, drow(seq, k), sd.x, inv_t, V, u, lane, tj, wt, wd);
        const df at = warp_sum_ordered(df_add(wt[0], wt[1]), lane);
        // p > q  <=>  e_t S_d > e_d S_t; the fp32 sums are good to well inside kSignBand
        df pt = df_zero(), pd = df_zero();
        int near = 0;
#pragma unroll
        for (int q = 0; q < kLane; ++q) {
            const float av = __fmul_rn(wt[q].hi, sd.y), bv = __fmul_rn(wd[q].hi, st.y);
            if (av > bv * (1.f + kSignBand)) {
                pt = df_add(pt, wt[q]);
                pd = df_add(pd, wd[q]);
            } else if (!(av < bv * (1.f - kSignBand)) && av > 0.f) {
                ++near;
            }
        }
        const df ad = warp_sum_ordered(df_add(wd[0], wd[1]), lane);
        pt = warp_sum_ordered(pt, lane);
        pd = warp_sum_ordered(pd, lane);
        near = warp_reduce(near, [](int x, int y) { return x + y; });
        if (lane == 0) {
            st_df(S + u, at);
            st_df(S + nu + u, ad);
            st_df(S + 2 * nu + u, pt);
            st_df(S + 3 * nu + u, pd);
            a.ramb[int64_t(e) * nu + u] = near;
        }
    }
    if (!barrier()) return;

    // F: one CTA per main-list sequence, the draw.
    for (int e = blockIdx.x; e < nmain; e += gridDim.x) {
        if (!SV_IN(e, B)) continue;  // (uniform over the CTA)
        const RefineInfo info = ldcg_info(a.rinfo + e);
        const int64_t seq = info.seq;
        if (!SV_IN(seq, B) || !SV_IN(info.k, gamma + 1)) continue;
        const int k = info.k;
        const df *S = a.rsum + e * slot;
        df *fix = a.rsum + e * slot + 4 * int64_t(nu);
        const int *near = a.ramb + int64_t(e) * nu;
        const float u2 = uniform01(a.seed, a.offset, uint32_t(seq), uint32_t(k), 1u);
        const float2 st = make_float2(info.Mt, info.St);
        auto all_t = [&](int q) { return ldcg_df(S + q); };
        df total, thr, b0;
        bool force;
        int tok = -1;
        if (info.mode == 1) {
            const float2 sd = make_float2(info.Md, info.Sd);
            df St, Sd;
            block_sum2(nu, all_t, [&](int q) { return ldcg_df(S + nu + q); }, &St, &Sd, sm);
            const df rho = df_div(St, Sd);
            // the near logits' exact residual weights, unit by unit (warps over the flagged
            // units; a warp reads the counts of kBatch groups of 32 units at once)
            for (int g0 = warp * 32; g0 < nu; g0 += kWarps * 32 * kBatch) {
                int cnt[kBatch];
#pragma unroll
                for (int q = 0; q < kBatch; ++q) {
                    const int uu = g0 + q * kWarps * 32 + lane;
                    cnt[q] = uu < nu ? __ldcg(near + uu) : 0;
                }
#pragma unroll 1
                for (int q = 0; q < kBatch; ++q) {
                    unsigned m = __ballot_sync(0xFFFFFFFFu, cnt[q] > 0);
                    while (m) {
                        const int u = g0 + q * kWarps * 32 + __ffs(m) - 1;
                        m &= m - 1;
                    df wt[kLane], wd[kLane];
                    lane_exps2<D>(trow(seq, k), st.x, drow(seq, k), sd.x, inv_t, V, u, lane, tj, wt, wd);
                    df fx = df_zero();
#pragma unroll
                    for (int q = 0; q < kLane; ++q) {
                        const float av = __fmul_rn(wt[q].hi, sd.y), bv = __fmul_rn(wd[q].hi, st.y);
                        if (!(av > bv * (1.f + kSignBand)) && !(av < bv * (1.f - kSignBand)) && av > 0.f)
                            fx = df_add(fx, resid(wt[q], wd[q], rho));
                    }
                    fx = warp_sum_ordered(fx, lane);
                    if (lane == 0) st_df(fix + u, fx);
                    }
                }
            }
            __syncthreads();
            const int u = block_search(
                nu, u2,
                [&](int q) {
                    df m = df_sub(ldcg_df(S + 2 * nu + q), df_mul(rho, ldcg_df(S + 3 * nu + q)));
                    return __ldcg(near + q) > 0 ? df_add(m, ldcg_df(fix + q)) : m;
                },
                &total, &thr, &b0, &force, sm);
            if (df_pos(total)) tok = pick(seq, k, st.x, sd.x, rho, true, u, b0, thr, force);
        }
        if (tok < 0 && info.mode == 2) {  // p without the token a one-hot q put all its mass on
            const int ex = a.x[seq * gamma + k], ex_u = ex / kUnit;
            const df ex_w = weight_df(load_elem<D>(trow(seq, k), ex), st.x, inv_t);
            const int u = block_search(
                nu, u2, [&](int q) { return q == ex_u ? df_sub(all_t(q), ex_w) : all_t(q); }, &total, &thr, &b0, &force,
                sm);
            if (df_pos(total)) tok = pick(seq, k, st.x, 0.f, df_zero(), false, u, b0, thr, force, ex);
        }
        if (tok < 0) {  // a bonus draw, or no residual mass at all: the draw from p on row k
            const int u = block_search(nu, u2, all_t, &total, &thr, &b0, &force, sm);
            tok = pick(seq, k, st.x, 0.f, df_zero(), false, u, b0, thr, force);
        }
        if (tid == 0) finish(seq, k, tok);
        __syncthreads();
    }
}

}  // namespace sv
