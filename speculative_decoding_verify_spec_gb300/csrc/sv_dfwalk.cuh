// sv_dfwalk.cuh -- warp-level building blocks of the double-float re-draws: the exponentials
// of one 256-logit unit, and inverse-CDF searches over stored unit sums.
//
// A unit is 256 consecutive logits of one row, lane l of the warp owning the contiguous
// logits [8 l, 8 l + 8).  Every sum over a unit is formed the same way -- a running DfSum
// per lane in index order, then an inclusive warp scan in lane order -- so the prefix that
// an in-unit scan reaches at the unit's end equals the stored unit sum bit for bit.
#pragma once

#include "sv_device.cuh"
#include "sv_df.cuh"

namespace sv {

constexpr int kDfUnit = 256;               // logits per unit (one warp)
constexpr int kDfLane = kDfUnit / 32;      // logits per lane, contiguous

__host__ __device__ inline int df_units(int V) { return int((int64_t(V) + kDfUnit - 1) / kDfUnit); }

__device__ __forceinline__ df ldcg_df(const df *p) {
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(p));
    return df{v.x, v.y};
}
__device__ __forceinline__ void st_df(df *p, df v) { *reinterpret_cast<float2 *>(p) = make_float2(v.hi, v.lo); }
__device__ __forceinline__ df df_zero() { return df{0.f, 0.f}; }

// max(e_t - ar e_d, 0): the residual weight (p - q)+ in units of S_t, with ar = a S_t / S_d.
__device__ __forceinline__ df resid_w(df et, df ed, df ar) {
    const df w = df_sub(et, df_mul(ar, ed));
    return df_pos(w) ? w : df_zero();
}

// The unit sum of per-logit values w (this lane's kDfLane of them, in index order, zero past
// the row's end): every lane returns the same value.
__device__ __forceinline__ df unit_sum(const df (&w)[kDfLane], int lane) {
    DfSum ls;
#pragma unroll
    for (int e = 0; e < kDfLane; ++e) ls.add(w[e]);
    return df_shfl(df_warp_scan(ls.value(), lane), 31);
}

// The double-float exponentials run rarely (only for the sequences an fp32 pass marked), so
// their code is not in the instruction cache when they do: every copy of it is fetched from
// L2 as it executes.  They are therefore kept out of line -- one copy of the eight-wide
// exponential and one of the single one, shared by every caller -- instead of being
// inlined and unrolled at each call site.
//
// w[e] = exp((x[e] - M) / T) for kDfLane logits, two independent chains interleaved at a
// time (a quarter of the code of all eight, which a cold instruction cache fetches faster).
static __device__ __noinline__ void weights_df(const float *x, float M, df inv_t, df *w) {
#pragma unroll 2
    for (int e = 0; e < kDfLane; ++e) w[e] = weight_df(x[e], M, inv_t);
}
// exp((x - M) / T) for one logit.
static __device__ __noinline__ df weight1_df(float x, float M, df inv_t) { return weight_df(x, M, inv_t); }

// exp((x_j - M) / T) of unit u of a row for this lane's logits (the loads first, all in
// flight together); 0 past the row's end.
template <class D>
__device__ __forceinline__ void unit_exps(const char *row, float M, df inv_t, int V, int u, int lane,
                                          df (&w)[kDfLane]) {
    const int64_t j0 = int64_t(u) * kDfUnit + lane * kDfLane;
    float x[kDfLane];
#pragma unroll
    for (int e = 0; e < kDfLane; ++e) x[e] = j0 + e < V ? load_elem<D>(row, j0 + e) : -__int_as_float(0x7f800000);
    weights_df(x, M, inv_t, w);
}

// Entry i of a list of n double-float values at vals[i * stride]; entry ex_i (if >= 0) is
// read as vals[ex_i] - ex_v (a unit sum without one excluded term).
__device__ __forceinline__ df df_entry(const df *vals, int stride, int i, int ex_i, df ex_v) {
    const df v = ldcg_df(vals + int64_t(i) * stride);
    return i == ex_i ? df_sub(v, ex_v) : v;
}

constexpr int kDfBatch = 8;  // values a lane loads together before it adds them (L2 latency)

// This lane's run of values [lane * per, (lane + 1) * per) of a list of n: the sum in index
// order and the index of the last positive one (-1 if none).
__device__ __forceinline__ df lane_run_sum(const df *vals, int stride, int n, int per, int lane, int ex_i, df ex_v,
                                           int *lastpos) {
    df ls = df_zero();
    for (int q0 = 0; q0 < per; q0 += kDfBatch) {
        df v[kDfBatch];
#pragma unroll
        for (int q = 0; q < kDfBatch; ++q) {
            const int i = lane * per + q0 + q;
            v[q] = (q0 + q < per && i < n) ? df_entry(vals, stride, i, ex_i, ex_v) : df_zero();
        }
#pragma unroll
        for (int q = 0; q < kDfBatch; ++q) {
            const int i = lane * per + q0 + q;
            if (q0 + q < per && i < n) {
                ls = df_add(ls, v[q]);
                if (df_pos(v[q])) *lastpos = i;
            }
        }
    }
    return ls;
}

// Warp-level search over n values in index order: the first i with base + vals[0] + ... +
// vals[i] > thr (lanes own contiguous runs: a lane prefix, then the lane's own run);
// *run_out = the prefix before i.  With no crossing (rounding left thr at or above the sum)
// or `force` set: the last i with a positive value and *force_out = true (-1 if every value
// is 0).  Every lane returns the same.
static __device__ __noinline__ int warp_search(const df *vals, int stride, int n, df base, df thr, bool force, df *run_out,
                                  bool *force_out, int lane, int ex_i = -1, df ex_v = df{0.f, 0.f}) {
    const int per = (n + 31) / 32;
    int lastpos = -1;
    const df ls = lane_run_sum(vals, stride, n, per, lane, ex_i, ex_v, &lastpos);
    if (!force) {
        const df incl = df_warp_scan(ls, lane);
        df excl = df_shfl_up(incl, 1);
        if (lane == 0) excl = df_zero();
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, df_gt(df_add(base, incl), thr));
        if (bal) {
            const int l = __ffs(bal) - 1;
            int found = -1;
            df run = df_add(base, excl);
            if (lane == l) {
                for (int q0 = 0; q0 < per && found < 0; q0 += kDfBatch) {
                    df v[kDfBatch];
#pragma unroll
                    for (int q = 0; q < kDfBatch; ++q) {
                        const int i = lane * per + q0 + q;
                        v[q] = (q0 + q < per && i < n) ? df_entry(vals, stride, i, ex_i, ex_v) : df_zero();
                    }
#pragma unroll
                    for (int q = 0; q < kDfBatch; ++q) {
                        const int i = lane * per + q0 + q;
                        if (found < 0 && q0 + q < per && i < n) {
                            const df nx = df_add(run, v[q]);
                            if (df_gt(nx, thr)) found = i;
                            else run = nx;
                        }
                    }
                }
            }
            found = __shfl_sync(0xFFFFFFFFu, found, l);
            run = df_shfl(run, l);
            if (found >= 0) {
                *run_out = run;
                *force_out = false;
                return found;
            }
        }
    }
    *run_out = df_zero();
    *force_out = true;
    return warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
}

// The sum of n values in warp_search's order (every lane returns it).
static __device__ __noinline__ df warp_total(const df *vals, int stride, int n, int lane, int ex_i = -1,
                                df ex_v = df{0.f, 0.f}) {
    const int per = (n + 31) / 32;
    int lastpos = -1;
    const df ls = lane_run_sum(vals, stride, n, per, lane, ex_i, ex_v, &lastpos);
    return df_shfl(df_warp_scan(ls, lane), 31);
}

// Inside the unit the search chose: the first logit whose prefix (run + this unit's values
// before it, inclusive) exceeds thr.  w: this lane's values of the unit (index order); j0:
// the index of this lane's first logit.  Rounding past the crossing lane's end, or `force`:
// the last logit with a positive value (the unit's first logit if none).  Every lane
// returns the same.
static __device__ __noinline__ int unit_pick(const df (&w)[kDfLane], int64_t unit0, int64_t j0, int V, df run, df thr, bool force,
                                int lane) {
    DfSum lsum;
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < kDfLane; ++e) {
        lsum.add(w[e]);
        if (j0 + e < V && df_pos(w[e])) lastpos = int(j0) + e;
    }
    lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
    int tok = lastpos;
    if (!force) {
        const df incl = df_warp_scan(lsum.value(), lane);
        df excl = df_shfl_up(incl, 1);
        if (lane == 0) excl = df_zero();
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, df_gt(df_add(run, incl), thr));
        if (bal) {
            const int l = __ffs(bal) - 1;
            int cand = -1, lpos = -1;
            df r2 = df_add(run, excl);
#pragma unroll
            for (int e = 0; e < kDfLane; ++e) {
                const df nx = df_add(r2, w[e]);
                if (cand < 0 && j0 + e < V && df_gt(nx, thr)) cand = int(j0) + e;
                if (j0 + e < V && df_pos(w[e])) lpos = int(j0) + e;
                r2 = nx;
            }
            if (cand < 0) cand = lpos;
            cand = __shfl_sync(0xFFFFFFFFu, cand, l);
            if (cand >= 0) tok = cand;
        }
    }
    if (tok < 0) tok = int(unit0);
    return tok;
}

}  // namespace sv
