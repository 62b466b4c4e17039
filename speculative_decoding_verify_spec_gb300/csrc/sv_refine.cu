// sv_refine.cu -- the extended-precision re-draw of near-boundary sampling sequences.
//
// The sampler's decisions are comparisons of sums of exponentials: u q(x) < p(x) for an
// accept test, C_j > u' R for the inverse CDF (first page, "The rule"; R3 of the readings).
// In fp32 a comparison whose two sides differ by less than ~1e-7 relative can come out the
// other way than in exact arithmetic.  decide and draw mark such sequences (margins below
// kRefineAcceptWindow / kRefineCdfWindow, far above the fp32 error) and this kernel redoes
// them in double-float arithmetic (sv_df.cuh, ~48 bits), which resolves every comparison
// whose exact margin is above ~1e-13.
//
// One cooperative grid (every CTA resident; launched behind draw like the other kernels of
// the call), two stages separated by a bounded grid barrier:
//   A  every 64-logit unit of the row pairs a listed sequence needs (its stop row k of
//      target and draft; every pair if an accept test was marked; target row gamma for a
//      bonus draw), one warp each: the unit sums of exp((x - M)/T) of both rows (M the row's
//      exact maximum) and the same sums over the logits where p - q is positive for certain
//      given the fp32 row sums (the sign of p - q is that of w_t S_d - w_d S_t); logits
//      within a 2e-6 band of that ratio go to a short ambiguity list;
//   B  one CTA per listed sequence: the row sums S; after a marked accept test the scan
//      again (p(x) = exp((x - M)/T) / S), rewriting accepted_len and the accepted prefix;
//      the unit masses of the final draw (sum+ w_t / S_t - sum+ w_d / S_d plus the listed
//      logits' (p - q)+, or sum w_t / S_t for p); a block scan finds the unit holding u' R,
//      one warp the first j with C_j > u' R inside it.
// The units are small (two logits per lane) because double-float arithmetic is a long
// dependent chain: wall time is the latency of one unit, so many units run at once.
// With nothing listed every CTA returns at once.
#include "spec_verify.h"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_grid.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kRefLane = 2;             // logits per lane in a re-draw unit
constexpr int kRefUnit = 32 * kRefLane;  // 64 logits per unit (one warp)
constexpr int kRefBatch = 8;             // loads issued together in the per-sequence stage
constexpr float kSignBand = 2e-6f;       // relative band around S_t / S_d left to the exact pass

// Block-wide double-float sum / inclusive scan (kThreads threads, index order = thread
// order).  `sm` holds kWarps values.
__device__ df block_df_sum(df v, df *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = df_warp_sum(v);
    __syncthreads();
    if (lane == 0) sm[warp] = v;
    __syncthreads();
    df t = sm[0];
    for (int w = 1; w < kWarps; ++w) t = df_add(t, sm[w]);
    return t;
}
__device__ df block_df_scan(df v, df *sm, df *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const df incl = df_warp_scan(v, lane);
    __syncthreads();
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    df before{0.f, 0.f}, all{0.f, 0.f};
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before = df_add(before, sm[w]);
        all = df_add(all, sm[w]);
    }
    *total = all;
    return df_add(before, incl);
}

// Per-sequence scratch (one slot per listed sequence), in units of nref entries:
//   all_t [gamma + 1][nref]  sum of exp((x - M)/T) over the unit, target rows
//   all_d [gamma][nref]      the same, draft rows
//   pos_t, pos_d [gamma][nref]  the same over the unit's logits where p - q is clearly > 0
// then per row pair an ambiguity list: count + kMaxAmbiguous positions.
struct Slot {
    df *base;
    int *amb;
    int gamma, nref;
    __device__ df *all_t(int r) const { return base + int64_t(r) * nref; }
    __device__ df *all_d(int i) const { return base + int64_t(gamma + 1 + i) * nref; }
    __device__ df *pos_t(int i) const { return base + int64_t(2 * gamma + 1 + i) * nref; }
    __device__ df *pos_d(int i) const { return base + int64_t(3 * gamma + 1 + i) * nref; }
    __device__ int *amb_list(int i) const { return amb + i * (1 + kMaxAmbiguous); }
};

// r = max(p - q, 0) of one logit pair, exactly (double-float), with the row sums known.
__device__ __forceinline__ df residual_df(float xt, float xd, float Mt, float Md, df inv_t, df inv_st, df inv_sd) {
    df w = df_sub(df_mul(weight_df(xt, Mt, inv_t), inv_st), df_mul(weight_df(xd, Md, inv_t), inv_sd));
    return df_pos(w) ? w : df{0.f, 0.f};
}

constexpr int kUnitsPerThread = 8;  // unit masses a thread of stage B keeps in registers

template <class D>
__global__ void __launch_bounds__(kThreads, 2)
    refine_kernel(Logits t, Logits d, int gamma, int V, int nref, float T, uint64_t seed, uint64_t offset,
                  const int32_t *__restrict__ x, const float2 *__restrict__ rowstat, int *__restrict__ rctl,
                  const RefineInfo *__restrict__ rinfo, df *__restrict__ rsum, int *__restrict__ ramb,
                  int32_t *__restrict__ accepted_len, int32_t *__restrict__ out_tokens) {
    __shared__ df sm[kWarps];
    __shared__ df sincl[kThreads];
    __shared__ df s_amb_r[kMaxAmbiguous];
    __shared__ int s_amb_u[kMaxAmbiguous];
    __shared__ int sh_unit, sh_first, sh_k;
    __shared__ df sh_base;
    griddep_launch_next();
    griddep_wait();
    const int listed = __ldcg(rctl + kRefineCount);
    const int count = listed < kMaxRefine ? listed : kMaxRefine;
    if (count == 0) return;  // the same for every CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    const int64_t nw = int64_t(gridDim.x) * kWarps;
    const int R = 2 * gamma + 1;
    const df inv_t = df_div(df_from(1.f), df_from(T));
    auto slot = [&](int j) {
        return Slot{rsum + int64_t(j) * slot_df_entries(gamma, nref), ramb + int64_t(j) * slot_amb_ints(gamma), gamma,
                    nref};
    };
    auto trow = [&](int64_t seq, int r) { return row_ptr(t, D::kBytes, seq, r); };
    auto drow = [&](int64_t seq, int i) { return row_ptr(d, D::kBytes, seq, i); };

    // A (all warps, one 64-logit unit each): for the row pairs a listed sequence needs --
    // its stop row k after a rejection, every pair after a marked accept test -- the unit
    // sums of exp((x - M)/T) of both rows, and of both rows over the logits where p > q
    // for certain given the fp32 row sums; logits inside the band go to the pair's
    // ambiguity list (draw cleared its count).  Target row gamma alone (bonus draw) only
    // needs its unit sums.
    for (int j = 0; j < count; ++j) {
        const RefineInfo info = rinfo[j];
        const int64_t seq = info.seq;
        const bool all = info.flag == kRefineAccept;
        const int k = info.k;
        const Slot sl = slot(j);
        const int p_lo = all ? 0 : (k < gamma ? k : 0), p_hi = all ? gamma : (k < gamma ? k + 1 : 0);
        const bool single = all || k == gamma;  // target row gamma alone
        const int rows = (p_hi - p_lo) + (single ? 1 : 0);
        const int64_t items = int64_t(rows) * nref;
        for (int64_t it = gw; it < items; it += nw) {
            const int ri = int(it / nref), u = int(it - int64_t(ri) * nref);
            const int64_t e0 = int64_t(u) * kRefUnit + lane * kRefLane;
            if (ri < p_hi - p_lo) {  // a row pair
                const int i = p_lo + ri;
                float2 st = make_float2(info.Mt, info.St), sd = make_float2(info.Md, info.Sd);
                if (all) {
                    st = rowstat[seq * R + i];
                    sd = rowstat[seq * R + gamma + 1 + i];
                }
                const char *tp = trow(seq, i), *dp = drow(seq, i);
                float xt[kRefLane], xd[kRefLane];
#pragma unroll
                for (int e = 0; e < kRefLane; ++e) {
                    xt[e] = e0 + e < V ? load_elem<D>(tp, e0 + e) : -__int_as_float(0x7f800000);
                    xd[e] = e0 + e < V ? load_elem<D>(dp, e0 + e) : -__int_as_float(0x7f800000);
                }
                df at{0.f, 0.f}, ad{0.f, 0.f}, pt{0.f, 0.f}, pd{0.f, 0.f};
#pragma unroll
                for (int e = 0; e < kRefLane; ++e) {
                    const df wt = weight_df(xt[e], st.x, inv_t);
                    const df wd = weight_df(xd[e], sd.x, inv_t);
                    at = df_add(at, wt);
                    ad = df_add(ad, wd);
                    // p > q  <=>  w_t S_d > w_d S_t; the fp32 sums are good to ~3.5e-7
                    const float a = __fmul_rn(wt.hi, sd.y), b = __fmul_rn(wd.hi, st.y);
                    if (a > b * (1.f + kSignBand)) {
                        pt = df_add(pt, wt);
                        pd = df_add(pd, wd);
                    } else if (!(a < b * (1.f - kSignBand)) && a > 0.f) {
                        int *list = sl.amb_list(i);
                        const int n = atomicAdd(list, 1);
                        if (n < kMaxAmbiguous) list[1 + n] = int(e0 + e);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {  // the four sums in one butterfly
                    at = df_add(at, df_shfl_xor(at, o));
                    ad = df_add(ad, df_shfl_xor(ad, o));
                    pt = df_add(pt, df_shfl_xor(pt, o));
                    pd = df_add(pd, df_shfl_xor(pd, o));
                }
                if (lane == 0) {
                    sl.all_t(i)[u] = at;
                    sl.all_d(i)[u] = ad;
                    sl.pos_t(i)[u] = pt;
                    sl.pos_d(i)[u] = pd;
                }
            } else {  // target row gamma
                const float M = all ? rowstat[seq * R + gamma].x : info.Mt;
                const char *tp = trow(seq, gamma);
                float xt[kRefLane];
#pragma unroll
                for (int e = 0; e < kRefLane; ++e) xt[e] = e0 + e < V ? load_elem<D>(tp, e0 + e) : -__int_as_float(0x7f800000);
                df at{0.f, 0.f};
#pragma unroll
                for (int e = 0; e < kRefLane; ++e) at = df_add(at, weight_df(xt[e], M, inv_t));
                at = df_warp_sum(at);
                if (lane == 0) sl.all_t(gamma)[u] = at;
            }
        }
    }
    if (!grid_barrier(rctl)) return;

    // B (one CTA per listed sequence): row sums, the accept scan again where decide marked
    // it, the unit masses of the final draw, the unit holding u' R and the token inside it
    for (int j = blockIdx.x; j < count; j += gridDim.x) {
        const RefineInfo info = rinfo[j];
        const int64_t seq = info.seq;
        const bool all = info.flag == kRefineAccept;
        const Slot sl = slot(j);
        // sums of one or two unit-sum arrays over all units, in one block reduction
        auto row_sums = [&](const df *a, const df *b, df *sa, df *sb) {
            df va{0.f, 0.f}, vb{0.f, 0.f};
            for (int u0 = threadIdx.x; u0 < nref; u0 += kThreads * kRefBatch) {
                df ea[kRefBatch], eb[kRefBatch];
#pragma unroll
                for (int q = 0; q < kRefBatch; ++q) {
                    const int u = u0 + q * kThreads;
                    ea[q] = u < nref ? a[u] : df{0.f, 0.f};
                    eb[q] = (b && u < nref) ? b[u] : df{0.f, 0.f};
                }
#pragma unroll
                for (int q = 0; q < kRefBatch; ++q) {
                    va = df_add(va, ea[q]);
                    vb = df_add(vb, eb[q]);
                }
            }
            *sa = block_df_sum(va, sm);
            if (b) *sb = block_df_sum(vb, sm);
        };
        int k2 = info.k, mode2 = info.mode;
        if (all) {  // every row's sum, then the scan in double-float, test by test
            k2 = gamma;
            for (int i = 0; i < gamma; ++i) {
                df St, Sd;
                row_sums(sl.all_t(i), sl.all_d(i), &St, &Sd);
                if (threadIdx.x == 0) {
                    const int32_t xi = x[seq * gamma + i];
                    const df p = df_div(weight_df(load_elem<D>(trow(seq, i), xi), rowstat[seq * R + i].x, inv_t), St);
                    const df q =
                        df_div(weight_df(load_elem<D>(drow(seq, i), xi), rowstat[seq * R + gamma + 1 + i].x, inv_t), Sd);
                    const float uu = uniform01(seed, offset, uint32_t(seq), uint32_t(i), 0u);
                    sh_k = df_lt(df_mul_f(q, uu), p) ? -1 : i;
                }
                __syncthreads();
                const int rej = sh_k;
                __syncthreads();
                if (rej >= 0) {
                    k2 = rej;
                    break;
                }
            }
            mode2 = k2 < gamma ? 1 : 0;
            if (warp == 0) {
                int32_t *out = out_tokens + seq * (gamma + 1);
                for (int i = lane; i <= gamma; i += 32) {
                    if (i < k2) out[i] = x[seq * gamma + i];
                    else if (i > k2) out[i] = -1;
                }
                if (lane == 0) accepted_len[seq] = k2;
            }
        }
        // the final draw's row sums (target; draft after a rejection)
        df St, Sd{1.f, 0.f};
        row_sums(sl.all_t(k2), mode2 ? sl.all_d(k2) : nullptr, &St, &Sd);
        const df inv_st = df_div(df_from(1.f), St), inv_sd = df_div(df_from(1.f), Sd);
        const float Mt = all ? rowstat[seq * R + k2].x : info.Mt;
        const float Md = mode2 ? (all ? rowstat[seq * R + gamma + 1 + k2].x : info.Md) : 0.f;
        const char *tp = trow(seq, k2), *dp = mode2 ? drow(seq, k2) : tp;
        // the ambiguous logits of the pair, exactly
        int namb = 0;
        if (mode2) {
            const int *list = sl.amb_list(k2);
            namb = list[0];
            if (namb > kMaxAmbiguous) namb = -1;  // too many to track: keep the fp32 draw
            if (namb > 0 && int(threadIdx.x) < namb) {
                const int jj = list[1 + threadIdx.x];
                s_amb_u[threadIdx.x] = jj / kRefUnit;
                s_amb_r[threadIdx.x] =
                    residual_df(load_elem<D>(tp, jj), load_elem<D>(dp, jj), Mt, Md, inv_t, inv_st, inv_sd);
            }
        }
        __syncthreads();
        if (namb < 0) continue;  // (uniform)
        // unit masses: thread t owns units [t per, (t + 1) per), the first kUnitsPerThread
        // of them kept in registers
        const int per = (nref + kThreads - 1) / kThreads;
        auto unit_mass = [&](int u, bool residual) {
            df m;
            if (residual) {
                m = df_sub(df_mul(sl.pos_t(k2)[u], inv_st), df_mul(sl.pos_d(k2)[u], inv_sd));
                for (int a = 0; a < namb; ++a)
                    if (s_amb_u[a] == u) m = df_add(m, s_amb_r[a]);
            } else {
                m = df_mul(sl.all_t(k2)[u], inv_st);
            }
            return m;
        };
        bool residual = mode2 == 1;
        df mine[kUnitsPerThread];
        df ls{0.f, 0.f}, total{0.f, 0.f}, incl{0.f, 0.f};
        for (int pass = 0; pass < 2; ++pass) {
            ls = df{0.f, 0.f};
            {  // the first kUnitsPerThread units: loads first, all together, then the arithmetic
                df a_[kUnitsPerThread], b_[kUnitsPerThread];
                const df *pa = residual ? sl.pos_t(k2) : sl.all_t(k2);
                const df *pb = sl.pos_d(k2);
#pragma unroll
                for (int q = 0; q < kUnitsPerThread; ++q) {
                    const int u = threadIdx.x * per + q;
                    const bool in = q < per && u < nref;
                    a_[q] = in ? pa[u] : df{0.f, 0.f};
                    b_[q] = (in && residual) ? pb[u] : df{0.f, 0.f};
                }
#pragma unroll
                for (int q = 0; q < kUnitsPerThread; ++q)
                    mine[q] = residual ? df_sub(df_mul(a_[q], inv_st), df_mul(b_[q], inv_sd)) : df_mul(a_[q], inv_st);
                if (residual && namb > 0) {
                    for (int a = 0; a < namb; ++a) {
                        const int q = s_amb_u[a] - int(threadIdx.x) * per;
                        if (q >= 0 && q < per && q < kUnitsPerThread) {
#pragma unroll
                            for (int qq = 0; qq < kUnitsPerThread; ++qq)
                                if (qq == q) mine[qq] = df_add(mine[qq], s_amb_r[a]);
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kUnitsPerThread; ++q) ls = df_add(ls, mine[q]);
            for (int q = kUnitsPerThread; q < per; ++q) {
                const int u = threadIdx.x * per + q;
                if (u < nref) ls = df_add(ls, unit_mass(u, residual));
            }
            incl = block_df_scan(ls, sm, &total);
            if (residual && !df_pos(total)) residual = false;  // no residual mass: draw from p
            else break;
        }
        const float u2 = uniform01(seed, offset, uint32_t(seq), uint32_t(k2), 1u);
        const df thr = df_mul_f(total, u2);
        sincl[threadIdx.x] = incl;
        if (threadIdx.x == 0) {
            sh_first = kThreads;
            sh_unit = -1;
        }
        __syncthreads();
        if (df_gt(incl, thr)) atomicMin(&sh_first, int(threadIdx.x));
        __syncthreads();
        if (int(threadIdx.x) == sh_first) {
            df run = threadIdx.x > 0 ? sincl[threadIdx.x - 1] : df{0.f, 0.f};
            int unit = -1, last = threadIdx.x * per;
#pragma unroll
            for (int q = 0; q < kUnitsPerThread; ++q) {
                const int u = threadIdx.x * per + q;
                if (unit < 0 && q < per && u < nref) {
                    last = u;
                    const df nxt = df_add(run, mine[q]);
                    if (df_gt(nxt, thr)) unit = u;
                    else run = nxt;
                }
            }
            for (int q = kUnitsPerThread; q < per && unit < 0; ++q) {
                const int u = threadIdx.x * per + q;
                if (u >= nref) break;
                last = u;
                const df nxt = df_add(run, unit_mass(u, residual));
                if (df_gt(nxt, thr)) unit = u;
                else run = nxt;
            }
            sh_unit = unit >= 0 ? unit : last;  // rounding: stay inside this thread's units
            sh_base = run;
        }
        __syncthreads();
        int unit = sh_unit;
        df base = sh_base;
        bool force_last = false;
        if (unit < 0) {  // rounding left the threshold at or above the total: the last unit with mass
            int lp = -1;
            for (int q = 0; q < per; ++q) {
                const int u = threadIdx.x * per + q;
                if (u < nref && df_pos(unit_mass(u, residual))) lp = u;
            }
            if (lp >= 0) atomicMax(&sh_unit, lp);
            __syncthreads();
            unit = sh_unit >= 0 ? sh_unit : 0;
            base = df{0.f, 0.f};
            force_last = true;
        }
        if (warp == 0) {  // inside the unit: lane l owns its kRefLane logits
            const int64_t c0 = int64_t(unit) * kRefUnit;
            df w[kRefLane];
            df wsum{0.f, 0.f};
#pragma unroll
            for (int e = 0; e < kRefLane; ++e) {
                const int64_t jj = c0 + lane * kRefLane + e;
                w[e] = df{0.f, 0.f};
                if (jj < V) {
                    w[e] = residual ? residual_df(load_elem<D>(tp, jj), load_elem<D>(dp, jj), Mt, Md, inv_t, inv_st,
                                                  inv_sd)
                                    : df_mul(weight_df(load_elem<D>(tp, jj), Mt, inv_t), inv_st);
                }
                wsum = df_add(wsum, w[e]);
            }
            const df lincl = df_warp_scan(wsum, lane);
            df run = df_add(base, df_sub(lincl, wsum));
            int cand = kNoIndex, lastpos = -1;
#pragma unroll
            for (int e = 0; e < kRefLane; ++e) {
                const int64_t jj = c0 + lane * kRefLane + e;
                run = df_add(run, w[e]);
                if (jj < V) {
                    if (!force_last && cand == kNoIndex && df_gt(run, thr)) cand = int(jj);
                    if (df_pos(w[e])) lastpos = int(jj);
                }
            }
            cand = warp_reduce(cand, [](int a, int b) { return min(a, b); });
            lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
            int tok = cand != kNoIndex ? cand : lastpos;
            if (tok < 0) tok = int(c0);
            if (lane == 0) out_tokens[seq * (gamma + 1) + k2] = int32_t(tok);
        }
        __syncthreads();
    }
}

// Test hook of the bounded wait: one CTA meets the re-draw's grid barrier expecting
// `expected` arrivals; with more than one nobody else comes, the wait runs out after
// limit_ns and records SV_ERR_TIMEOUT in ctl[kBarStatus] (the same path a stalled re-draw
// takes).
__global__ void wait_selftest_kernel(int *ctl, int expected, uint64_t limit_ns) {
    if (threadIdx.x == 0) {
        ctl[kBarCount] = 0;
        ctl[kBarStatus] = 0;
    }
    __syncthreads();
    grid_barrier(ctl, expected, limit_ns);
}

__global__ void exp_df_kernel(const float *__restrict__ y_hi, const float *__restrict__ y_lo, int n,
                              float *__restrict__ out_hi, float *__restrict__ out_lo) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const df e = exp_df(df{y_hi[i], y_lo[i]});
    out_hi[i] = e.hi;
    out_lo[i] = e.lo;
}

}  // namespace

cudaError_t launch_refine(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V, int nref, float T,
                          uint64_t seed, uint64_t offset, const int32_t *x, const void *rowstat, const void *plan,
                          int *rctl, const RefineInfo *rinfo, void *rsum, void *ramb, int32_t *accepted_len,
                          int32_t *out_tokens, cudaStream_t s) {
    (void)B;
    (void)vec;   // element loads: any alignment
    (void)plan;  // the listed sequences' plans travel in their RefineInfo records
    auto k = dtype == 1 ? refine_kernel<BF16> : refine_kernel<F32>;
    // one CTA per SM (all resident, as the grid barrier needs): a step without a marked
    // sequence then spends less on launching and retiring it than with every resident slot
    // filled (measured 0.9 us per step), and a marked one about the same
    unsigned grid = 0;
    int dev = 0, sms = 0;
    cudaError_t e = persistent_grid(k, int64_t(1) << 40, &grid);
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms > 0 && grid > unsigned(sms)) grid = unsigned(sms);
    return launch_after_ex(true, k, grid, kThreads, 0, s, t, d, gamma, V, nref, T, seed, offset, x,
                           static_cast<const float2 *>(rowstat), rctl, rinfo, static_cast<df *>(rsum),
                           static_cast<int *>(ramb), accepted_len, out_tokens);
}

cudaError_t launch_wait_selftest(int *ctl, int expected, uint64_t limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(ctl, expected, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_exp_df(const float *y_hi, const float *y_lo, int n, float *out_hi, float *out_lo,
                          cudaStream_t s) {
    exp_df_kernel<<<unsigned((n + 255) / 256), 256, 0, s>>>(y_hi, y_lo, n, out_hi, out_lo);
    return cudaGetLastError();
}

}  // namespace sv
