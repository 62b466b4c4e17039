// sv_tree_sample.cu -- token-tree SAMPLING verification: multi-round (recursive) rejection.
//
// Method ("7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead", "Tree
// Attention: Verifying Many Candidates at Once", the paragraph on SpecInfer's rule): at an
// accepted node v the children are tested in order against the current (p, q) with the
// single-candidate rule; a rejection replaces p by the normalised residual (p - q)+ and,
// when the siblings were drawn without replacement, q by q without the rejected token,
// renormalised; when every child is rejected the final token comes from the last
// residual, at a leaf it is the bonus drawn from p at the leaf.
//
// The walk is sequential and data-dependent, so it runs lazily: one CTA per sequence
// reads only the rows of the nodes it reaches.  p and q are never materialised.  With
// p0 = softmax(t_v / T) and q0 = softmax(d_v / T), after r rejections
//     p_r(j) = w_r(j) / D_r,   w_r(j) = max(p0(j) - a_r(j) q0(j), 0),
//     q_r(j) = s_r q0(j)  (0 for a token removed from q),
// where a_r(j) = A_r for every token still in q and the value A had when the token was
// removed for the others.  A rejection at round r sets A_{r+1} = A_r + D_r s_r and
// D_{r+1} = sum_j w_{r+1}(j) (one pass over the row pair); without replacement s_{r+1} =
// 1 / (1 - the removed tokens' q0 mass).  (Induction on r: for a token still in q,
// p_r - q_r = (max(p0 - A_r q0, 0) - D_r s_r q0) / D_r, whose positive part is
// max(p0 - A_{r+1} q0, 0) / D_r.)  Each pass stores one mass per unit of res_tile_elems
// logits, and the final draw walks those masses and then one unit, as the chain's draw.
//
// Arithmetic mirrors the chain sampler: weights 2^((x - M) c) with x - M exact, explicitly
// rounded products, fp32 sums in a fixed order; the final draw's prefixes in fp64.
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTsThreads = 1024;
constexpr int kTsWarps = kTsThreads / 32;
constexpr int kMaxRemoved = 64;  // tokens removed from q at one node (without replacement)

__device__ __forceinline__ float tweight(float x, float M, float c) { return ex2(__fmul_rn(__fsub_rn(x, M), c)); }

// The state of the current node: its rows' statistics and the implicit (p, q).
struct NodeState {
    float Mt, inv_st, Md, inv_sd;  // (max, 1 / sum) of target row v and draft row v
    float A, Dn, s;                // a coefficient, D_r, q's scale
    float qrem;                    // removed tokens' q0 mass
    int nrem;                      // tokens removed from q
    bool has_q;                    // the draft row was read (v has children)
};

// w(j) of one logit pair under coefficient a (a = 0: p0 alone; the draft is not used).
__device__ __forceinline__ float wgt(float tj, float dj, const NodeState &s, float a, float c) {
    const float p = __fmul_rn(tweight(tj, s.Mt, c), s.inv_st);
    if (a == 0.f) return p;
    const float q = __fmul_rn(tweight(dj, s.Md, c), s.inv_sd);
    return fmaxf(__fsub_rn(p, __fmul_rn(a, q)), 0.f);
}

template <class D, bool VEC>
__device__ __forceinline__ void load_unit(const char *row, int64_t u0, int len, int lane, uint4 (&v)[kResVecs]) {
#pragma unroll
    for (int k = 0; k < kResVecs; ++k) {
        const int e0 = (lane + 32 * k) * D::EPV;
        v[k] = e0 < len ? load_vec<D, VEC>(row, u0, e0, len) : neg_inf_vec<D>();
    }
}

}  // namespace

// One cluster of CS CTAs per sequence: every CTA runs the same walk, takes every CS-th
// unit of each pass, and merges the CTAs' partials in rank order after a cluster barrier,
// so all of them take the same decisions; rank 0 draws and writes the outputs.  cstat:
// [B][CS][2] per-CTA row statistics.  Shared: parent, tokens, child counts, depths, the path, the
// removed tokens and their frozen coefficients, and the reduction scratch.
template <class D, bool VEC, int CS>
__global__ void __launch_bounds__(kTsThreads, 1)
    tree_sample_kernel(Logits t, Logits d, int N, int V, const int32_t *__restrict__ parent,
                       const int32_t *__restrict__ node_tokens, int max_depth, float c, uint64_t seed,
                       uint64_t offset, int without_replacement, int nunit, float *umass, float2 *cstat,
                       TreeRefineWs rw, int K, int32_t *__restrict__ accepted_len,
                       int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_path) {
    extern __shared__ int s_int[];
    int *s_par = s_int, *s_tok = s_int + N, *s_nch = s_int + 2 * N, *s_dep = s_int + 3 * N;
    int *s_path = s_int + 4 * N;  // max_depth + 1
    __shared__ int s_remtok[kMaxRemoved];
    __shared__ float s_remcoef[kMaxRemoved];
    __shared__ float2 s_stat[2][kTsWarps];
    __shared__ float s_sum[kTsWarps];
    __shared__ int s_flag;
    __shared__ int s_near;  // kTrMark* bits: a decision came near flipping in fp32 (the re-walk redoes it)
    __shared__ int s_nrec;  // nodes recorded for the re-walk
    __shared__ float s_tx[2];
    griddep_launch_next();
    griddep_wait();  // the caller's kernels may still be writing the inputs
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t seq = blockIdx.x / CS;
    const int rank = cluster_rank<CS>();
    const int gw = rank * kTsWarps + warp;  // this warp among the cluster's
    const int W = max_depth + 1;
    int32_t *out = out_tokens + seq * W;
    int32_t *opath = out_path ? out_path + seq * W : nullptr;
    float *um = umass + seq * int64_t(nunit);
    constexpr int RE = res_tile_elems<D>();

    if (blockIdx.x == 0) {  // the re-walk's control words and counters (it starts after this grid)
        if (tid < kTrCtlWords) rw.ctl[tid] = 0;
        for (int i = tid; i < kMaxTreeRefine * K; i += kTsThreads) rw.npos[i] = 0;
    }
    // the tree and the tokens: parent[0] = -1, parent[v] in [0, v), depth <= max_depth
    if (tid == 0) {
        s_flag = 1;
        s_near = 0;
        s_nrec = 0;
    }
    __syncthreads();
    for (int v = tid; v < N; v += kTsThreads) {
        const int p = parent[v];
        s_par[v] = p;
        s_nch[v] = 0;
        const int tk = v == 0 ? 0 : node_tokens[seq * N + v];
        s_tok[v] = tk;
        if ((v == 0 && p != -1) || (v > 0 && (p < 0 || p >= v)) || tk < 0 || tk >= V) s_flag = 0;
    }
    __syncthreads();
    if (s_flag) {
        for (int v = tid; v < N; v += kTsThreads) {
            int dpt = 0;
            for (int w = v; w != 0 && dpt <= max_depth; w = s_par[w]) ++dpt;
            s_dep[v] = dpt;
            if (dpt > max_depth) s_flag = 0;
            if (v > 0) atomicAdd(&s_nch[s_par[v]], 1);
        }
    }
    __syncthreads();
    auto fail = [&]() {
        if (rank != 0) return;
        for (int i = tid; i < W; i += kTsThreads) {
            out[i] = -1;
            if (opath) opath[i] = -1;
        }
        if (tid == 0) {
            accepted_len[seq] = -1;
            rw.mark[seq] = s_near;  // a near decision may have led to this row
            rw.rlen[seq] = s_nrec;
        }
    };
    if (!s_flag) {
        fail();
        return;
    }

    // One pass over the units of row pair v: every warp takes units warp, warp + 32, ...;
    // the unit masses go to um[], their total (fixed order) is returned to every thread.
    // a = 0 reads the target row only.
    auto mass_pass = [&](const char *tp, const char *dp, const NodeState &st, float a) -> float {
        for (int u = gw; u < nunit; u += CS * kTsWarps) {
            const int64_t u0 = int64_t(u) * RE;
            const int len = unit_len(V, u0, RE);
            uint4 tv[kResVecs], dv[kResVecs];
            load_unit<D, VEC>(tp, u0, len, lane, tv);
            if (a != 0.f) load_unit<D, VEC>(dp, u0, len, lane, dv);
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < kResVecs; ++k)
#pragma unroll
                for (int e = 0; e < D::EPV; ++e)
                    acc += wgt(vec_elem<D>(tv[k], e), a != 0.f ? vec_elem<D>(dv[k], e) : 0.f, st, a, c);
            acc = warp_reduce(acc, [](float x, float y) { return x + y; });
            if (lane == 0 && SV_IN(u, nunit)) um[u] = acc;
        }
        csync<CS>();  // the unit masses of every warp of the cluster
        // tokens removed earlier keep their own coefficient: correct their units (rank 0)
        bool fix = false;  // (the same in every thread of the cluster)
        if (a != 0.f)
            for (int r = 0; r < st.nrem; ++r) fix |= s_remcoef[r] != a;
        if (fix) {
            if (rank == 0 && tid == 0) {
                for (int r = 0; r < st.nrem; ++r) {
                    if (s_remcoef[r] == a) continue;
                    const int j = s_remtok[r];
                    const float tj = load_elem<D>(tp, j), dj = load_elem<D>(dp, j);
                    if (SV_IN(j / RE, nunit)) um[j / RE] += wgt(tj, dj, st, s_remcoef[r], c) - wgt(tj, dj, st, a, c);
                }
            }
            csync<CS>();
        }
        // total: lanes of warp 0 own contiguous runs of units, then a warp scan
        if (warp == 0) {
            const int per = (nunit + 31) / 32;
            float ls = 0.f;
            for (int q = 0; q < per; ++q) {
                const int u = lane * per + q;
                if (u < nunit) ls += um[u];
            }
            const float tot = __shfl_sync(0xFFFFFFFFu, warp_inclusive_scan(ls, lane), 31);
            if (lane == 0) s_sum[0] = tot;
        }
        __syncthreads();
        const float tot = s_sum[0];
        csync<CS>();  // every CTA has read um[] before any may start the next pass
        return tot;
    };

    // (max, sum) of the target row and, with two, of the draft row, in one pass (both rows'
    // loads in flight together): warps reduce units, then a fixed-order merge per row; every
    // thread returns the target row's (M, S) and *ds the draft row's ((0, 1) without two).
    auto row_stats2 = [&](const char *tp, const char *dp, bool two, float2 *ds) -> float2 {
        float2 wt = make_float2(-__int_as_float(0x7f800000), 0.f), wd = wt;
        for (int u = gw; u < nunit; u += CS * kTsWarps) {
            const int64_t u0 = int64_t(u) * RE;
            const int len = unit_len(V, u0, RE);
            uint4 vt[kResVecs], vd[kResVecs];
            load_unit<D, VEC>(tp, u0, len, lane, vt);
            if (two) load_unit<D, VEC>(dp, u0, len, lane, vd);
            const float Mt = warp_reduce(thread_max<D>(vt), [](float x, float y) { return max_nan(x, y); });
            float St = 0.f;
            if (is_finite(Mt)) St = warp_reduce(thread_sumexp<D>(vt, c, Mt), [](float x, float y) { return x + y; });
            wt = merge_stats(wt, make_float2(Mt, St), c);
            if (two) {
                const float Md = warp_reduce(thread_max<D>(vd), [](float x, float y) { return max_nan(x, y); });
                float Sd = 0.f;
                if (is_finite(Md)) Sd = warp_reduce(thread_sumexp<D>(vd, c, Md), [](float x, float y) { return x + y; });
                wd = merge_stats(wd, make_float2(Md, Sd), c);
            }
        }
        if (lane == 0) {
            s_stat[0][warp] = wt;
            s_stat[1][warp] = wd;
        }
        __syncthreads();
        float2 rt = s_stat[0][0], rd = s_stat[1][0];
        for (int w = 1; w < kTsWarps; ++w) {
            rt = merge_stats(rt, s_stat[0][w], c);
            rd = merge_stats(rd, s_stat[1][w], c);
        }
        if constexpr (CS > 1) {  // the CTAs' statistics, merged in rank order by each CTA
            float2 *cs = cstat + seq * CS * 2;
            if (tid == 0) {
                cs[rank * 2] = rt;
                cs[rank * 2 + 1] = rd;
            }
            csync<CS>();
            rt = cs[0];
            rd = cs[1];
            for (int k = 1; k < CS; ++k) {
                rt = merge_stats(rt, cs[k * 2], c);
                rd = merge_stats(rd, cs[k * 2 + 1], c);
            }
            csync<CS>();  // read by every CTA before the next statistics overwrite them
        } else {
            __syncthreads();
        }
        *ds = two ? rd : make_float2(0.f, 1.f);
        return rt;
    };

    int v = 0, depth = 0;
    if (tid == 0) s_path[0] = 0;
    NodeState st{};
    for (;;) {
        const char *tp = row_ptr(t, D::kBytes, seq, v);
        const char *dp = row_ptr(d, D::kBytes, seq, v);
        st.has_q = s_nch[v] > 0;
        float2 ds;
        const float2 ts = row_stats2(tp, dp, st.has_q, &ds);
        if (!is_finite(ts.x) || (st.has_q && !is_finite(ds.x))) {  // not a distribution (R11)
            fail();
            return;
        }
        if (rank == 0 && tid == 0 && depth < K && SV_IN(v, N)) {  // the node and its rows' maxima, for the re-walk
            rw.rec[seq * K + depth] = make_float4(__int_as_float(v), ts.x, st.has_q ? ds.x : 0.f, st.has_q ? 1.f : 0.f);
            s_nrec = depth + 1;
        }
        st.Mt = ts.x;
        st.inv_st = 1.f / ts.y;
        st.Md = ds.x;
        st.inv_sd = 1.f / ds.y;
        st.A = 0.f;
        st.Dn = 1.f;
        st.s = 1.f;
        st.qrem = 0.f;
        st.nrem = 0;
        bool residual_ready = false;  // um[] holds the masses of the current w
        float last_total = 0.f;       // ... and their total
        int next = -1;
        for (int cnode = v + 1; cnode < N && next < 0; ++cnode) {
            if (s_par[cnode] != v) continue;
            const int x = s_tok[cnode];
            if (tid == 0) {
                s_tx[0] = load_elem<D>(tp, x);
                s_tx[1] = load_elem<D>(dp, x);
            }
            __syncthreads();
            const float tx = s_tx[0], dx = s_tx[1];
            __syncthreads();
            // the current p(x) and q(x)
            float ax = st.A;
            bool removed = false;
            for (int r = 0; r < st.nrem; ++r)
                if (s_remtok[r] == x) {
                    ax = s_remcoef[r];
                    removed = true;
                }
            const float p0x = __fmul_rn(tweight(tx, st.Mt, c), st.inv_st);
            const float q0x = __fmul_rn(tweight(dx, st.Md, c), st.inv_sd);
            const float wx = ax == 0.f ? p0x : fmaxf(__fsub_rn(p0x, __fmul_rn(ax, q0x)), 0.f);
            const float px = wx / st.Dn;
            const float qx = removed ? 0.f : __fmul_rn(st.s, q0x);
            const float u = uniform01(seed, offset, uint32_t(seq), uint32_t(cnode - 1), 0u);
            const float uq = u * qx;
            // p's error: its own terms' rounding and D's, relative to D (both shrink with D)
            if (tid == 0 &&
                fabsf(uq - px) < kTreeAcceptWindow * (fmaxf(px, uq) + __fdividef(p0x + ax * q0x + px * st.A, st.Dn)))
                s_near |= kTrMarkPath;
            if (uq < px) {  // accepted
                next = cnode;
                break;
            }
            // rejected: A grows by D s (q's current scale), x leaves q without replacement
            const float Anew = __fadd_rn(st.A, __fmul_rn(st.Dn, st.s));
            NodeState ns = st;
            if (tid == 0 && without_replacement && !removed && st.nrem >= kMaxRemoved) s_near |= kTrMarkPath;
            if (without_replacement && !removed && st.nrem < kMaxRemoved) {
                if (tid == 0) {
                    s_remtok[st.nrem] = x;
                    s_remcoef[st.nrem] = Anew;
                }
                ns.nrem = st.nrem + 1;
                ns.qrem = __fadd_rn(st.qrem, q0x);
                ns.s = ns.qrem < 1.f ? 1.f / __fsub_rn(1.f, ns.qrem) : 0.f;
                if (tid == 0 && !(ns.qrem < 1.f - kTreeQMassWindow)) s_near |= kTrMarkPath;
            }
            __syncthreads();
            const float F = mass_pass(tp, dp, ns, Anew);
            if (tid == 0 && !(F > kTreeMassWindow * (1.f + Anew))) s_near |= kTrMarkPath;
            if (F > 0.f) {
                ns.A = Anew;
                ns.Dn = F;
                residual_ready = true;
                last_total = F;
            } else {  // no residual mass: p stays (the removal from q still happens)
                ns.A = st.A;
                ns.Dn = st.Dn;
                residual_ready = false;
                if (without_replacement && ns.nrem > st.nrem && tid == 0) s_remcoef[st.nrem] = st.A;
            }
            st = ns;
            __syncthreads();
        }
        if (next >= 0) {
            ++depth;
            if (!SV_IN(depth, W) || !SV_IN(next, N)) {  // (the same in every thread)
                fail();
                return;
            }
            if (tid == 0) s_path[depth] = next;
            v = next;
            continue;
        }
        // the final token at v: from w under the current state (the last residual, or p)
        const float total = residual_ready ? last_total : mass_pass(tp, dp, st, st.A);
        (void)total;
        if (warp == 0 && rank == 0) {
            // The prefixes and the threshold in double-float (sums of the fp32 weights good to
            // ~2^-48): the comparison is then limited by the weights' own rounding, not by the
            // resolution of an fp32 running sum, and near-boundary draws are rarer.
            const float u2 = uniform01(seed, offset, uint32_t(seq), uint32_t(v), 1u);
            const int per = (nunit + 31) / 32;
            PairSum lacc;
            for (int q = 0; q < per; ++q) {
                const int uu = lane * per + q;
                if (uu < nunit) lacc.add(um[uu]);
            }
            const df incl = df_warp_scan(lacc.value(), lane);
            const df totd = df_shfl(incl, 31);
            const df thr = df_mul_f(totd, u2);
            int unit = -1;
            df base = df{0.f, 0.f};
            bool force_last = false;
            const unsigned crossing = __ballot_sync(0xFFFFFFFFu, df_gt(incl, thr));
            if (crossing) {
                const int l = __ffs(crossing) - 1;
                df excl = df_shfl_up(incl, 1);
                if (lane == 0) excl = df{0.f, 0.f};
                if (lane == l) {
                    df run = excl;
                    int last_in_lane = lane * per;
                    for (int q = 0; q < per && unit < 0; ++q) {
                        const int uu = lane * per + q;
                        if (uu >= nunit) break;
                        last_in_lane = uu;
                        const df nx = df_add(run, df_from(um[uu]));
                        if (df_gt(nx, thr)) unit = uu;
                        else run = nx;
                    }
                    if (unit < 0) unit = last_in_lane;
                    base = run;
                }
                unit = __shfl_sync(0xFFFFFFFFu, unit, l);
                base = df_shfl(base, l);
            } else {  // rounding left the threshold at or above the total: the last unit with mass
                int lp = -1;
                for (int q = 0; q < per; ++q) {
                    const int uu = lane * per + q;
                    if (uu < nunit && um[uu] > 0.f) lp = uu;
                }
                lp = warp_reduce(lp, [](int a, int b) { return max(a, b); });
                unit = lp >= 0 ? lp : 0;
                force_last = true;
            }
            // inside the unit: lane l owns the contiguous vectors [l kResVecs, (l + 1) kResVecs)
            const int64_t u0 = int64_t(unit) * RE;
            const int len = unit_len(V, u0, RE);
            uint4 tv[kResVecs], dv[kResVecs];
#pragma unroll
            for (int k = 0; k < kResVecs; ++k) {
                const int e0 = (lane * kResVecs + k) * D::EPV;
                tv[k] = e0 < len ? load_vec<D, VEC>(tp, u0, e0, len) : neg_inf_vec<D>();
                dv[k] = (st.A != 0.f && e0 < len) ? load_vec<D, VEC>(dp, u0, e0, len) : neg_inf_vec<D>();
            }
            auto w_at = [&](int k, int e) -> float {
                const int j = int(u0) + (lane * kResVecs + k) * D::EPV + e;
                float a = st.A;
                for (int r = 0; r < st.nrem; ++r)
                    if (s_remtok[r] == j) a = s_remcoef[r];
                return wgt(vec_elem<D>(tv[k], e), st.A != 0.f ? vec_elem<D>(dv[k], e) : 0.f, st, a, c);
            };
            PairSum lsum;
            int lastpos = -1;
#pragma unroll
            for (int k = 0; k < kResVecs; ++k)
#pragma unroll
                for (int e = 0; e < D::EPV; ++e) {
                    const int j = (lane * kResVecs + k) * D::EPV + e;
                    const float w = w_at(k, e);
                    lsum.add(w);
                    if (j < len && w > 0.f) lastpos = j;
                }
            const df lincl = df_warp_scan(lsum.value(), lane);
            df lexcl = df_shfl_up(lincl, 1);
            if (lane == 0) lexcl = df{0.f, 0.f};
            // the lane whose run crosses thr, then its logits one per lane and a second scan
            constexpr int NE = kResVecs * D::EPV;  // logits per lane
            int first = kNoIndex;
            float gap = 0.f;  // distance of thr to the chosen token's CDF boundaries
            const unsigned lb = force_last ? 0u : __ballot_sync(0xFFFFFFFFu, df_gt(df_add(base, lincl), thr));
            if (lb) {
                const int l3 = __ffs(lb) - 1;
                const int j = l3 * NE + lane;
                float w = 0.f;
                if (lane < NE && j < len) {
                    float a = st.A;
                    for (int r = 0; r < st.nrem; ++r)
                        if (s_remtok[r] == int(u0) + j) a = s_remcoef[r];
                    w = wgt(load_elem<D>(tp, u0 + j), st.A != 0.f ? load_elem<D>(dp, u0 + j) : 0.f, st, a, c);
                }
                const df start = df_add(base, df_shfl(lexcl, l3));
                const df above = df_sub(df_add(start, df_warp_scan(df_from(w), lane)), thr);  // C_j - thr
                const unsigned eb = __ballot_sync(0xFFFFFFFFu, lane < NE && j < len && df_pos(above));
                if (eb) {
                    const int le = __ffs(eb) - 1;
                    first = l3 * NE + le;
                    const float ah = __shfl_sync(0xFFFFFFFFu, above.hi, le);
                    const float wl = __shfl_sync(0xFFFFFFFFu, w, le);
                    gap = fminf(__fsub_rn(wl, ah), ah);  // thr - C_{j-1} = w - (C_j - thr)
                }
            }
            // (p0's terms from target row v, A q0's from draft row v)
            const float win = kTreeCdfWindow * (totd.hi + st.A) + token_window(1.f / st.inv_st) +
                              (st.A != 0.f ? st.A * token_window(1.f / st.inv_sd) : 0.f);
            if (lane == 0 && (first == kNoIndex || force_last || !(gap >= win)))
                s_near |= kTrMarkFinal;
            lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
            int tok = first != kNoIndex ? first : lastpos;
            if (tok < 0) tok = 0;
            if (lane == 0) s_tx[0] = __int_as_float(int(u0) + tok);
        }
        __syncthreads();
        break;
    }
    if (rank != 0) return;
    if (tid == 0) {
        rw.mark[seq] = s_near;
        rw.rlen[seq] = s_nrec;
    }
    // outputs: the path (root .. v), its tokens, the final token, -1 padding
    const int tok = __float_as_int(s_tx[0]);
    for (int i = tid; i < W; i += kTsThreads) {
        int o = -1, pth = -1;
        if (i <= depth) pth = s_path[i];
        if (i < depth) o = SV_IN(s_path[i + 1], N) ? s_tok[s_path[i + 1]] : -1;
        else if (i == depth) o = tok;
        out[i] = o;
        if (opath) opath[i] = pth;
    }
    if (tid == 0) accepted_len[seq] = depth;
}

namespace {
template <int CS>
cudaError_t launch_walk(int dtype, bool vec, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                        const int32_t *node_tokens, int max_depth, float c, uint64_t seed, uint64_t offset,
                        int without_replacement, int nunit, float *umass, float2 *cstat, TreeRefineWs rw, int K,
                        int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path, cudaStream_t s) {
    const size_t smem = size_t(4 * N + max_depth + 1) * sizeof(int);
    auto k = dtype == 1 ? (vec ? tree_sample_kernel<BF16, true, CS> : tree_sample_kernel<BF16, false, CS>)
                        : (vec ? tree_sample_kernel<F32, true, CS> : tree_sample_kernel<F32, false, CS>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B) * CS);
    cfg.blockDim = dim3(kTsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CS > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, t, d, N, V, parent, node_tokens, max_depth, c, seed, offset,
                              without_replacement, nunit, umass, cstat, rw, K, accepted_len, out_tokens, out_path);
}
}  // namespace

// The cluster size: as many SMs per sequence as keep every sequence's cluster resident at
// once (a pass is a few unit loads per warp, so a second wave of clusters costs more than
// a wider cluster saves).
cudaError_t launch_tree_sample(int dtype, bool vec, Logits t, Logits d, int B, int N, int V,
                               const int32_t *parent, const int32_t *node_tokens, int max_depth, float c, uint64_t seed,
                               uint64_t offset, int without_replacement, int nunit, float *umass, float2 *cstat,
                               TreeRefineWs rw, int K, int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                               cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    static_assert(kTreeSampleCluster == 4, "the statistics scratch is sized for clusters of up to 4");
    if (int64_t(B) * 4 <= sms)
        return launch_walk<4>(dtype, vec, t, d, B, N, V, parent, node_tokens, max_depth, c, seed, offset,
                              without_replacement, nunit, umass, cstat, rw, K, accepted_len, out_tokens, out_path, s);
    if (int64_t(B) * 2 <= sms)
        return launch_walk<2>(dtype, vec, t, d, B, N, V, parent, node_tokens, max_depth, c, seed, offset,
                              without_replacement, nunit, umass, cstat, rw, K, accepted_len, out_tokens, out_path, s);
    return launch_walk<1>(dtype, vec, t, d, B, N, V, parent, node_tokens, max_depth, c, seed, offset,
                          without_replacement, nunit, umass, cstat, rw, K, accepted_len, out_tokens, out_path, s);
}

}  // namespace sv
