// sv_tree_refine.cu -- the extended-precision re-walk of near-boundary tree-sampling sequences.
//
// The walk (sv_tree_sample.cu) takes its decisions in fp32: accept tests u q(x) < p(x),
// residual masses and the inverse-CDF draw ("Tree Attention: Verifying Many Candidates at
// Once", SpecInfer's rule; "The rule" for the single test).  A comparison whose two sides
// lie closer than the fp32 error may come out the other way than in exact arithmetic, and
// every later decision depends on it, so the walk marks such a sequence and records the
// nodes it reached with their rows' maxima; these kernels walk every marked sequence
// (index order) again from the root in double-float arithmetic
// (sv_df.cuh, ~48 bits; the arithmetic of the chain's re-draw), which settles every
// comparison whose exact margin is above ~1e-12.
//
//   tree_exp_kernel     the whole grid (one cooperative launch): for every recorded node of
//                       the first eight marked sequences, e_t(j) = exp((t_j - M_t) / T) and
//                       e_d(j) of its target and draft rows, stored with their 256-logit unit
//                       sums and q's support size; then, for those of them marked only at
//                       their final draw (their path certain), the rejections at the reached
//                       node and the final draw again, every residual pass spread over the
//                       whole grid (slots in lock step, one grid barrier per pass);
//   tree_rewalk_kernel  eight thread-block clusters, each taking every eighth marked
//                       sequence in turn (the first one with those stored values, later ones
//                       computing them in the cluster), its CTAs owning
//                       contiguous runs of units and meeting at hardware cluster barriers:
//                       the rows' sums S_t, S_d, the child tests, one pass per rejection
//                       for the residual weights in S_t units
//                           W(j) = max(e_t(j) - a_j rho e_d(j), 0),   rho = S_t / S_d,
//                       (the walk's w(j) = max(p0(j) - a_j q0(j), 0) times S_t, a_j the
//                       coefficient of the walk's implicit form), and the final draw: the
//                       CTA run, then the unit, then the logit holding u' x total, each by a
//                       prefix in index order.  A node the walk did not record (the re-walk
//                       took another child) gets its maxima and exponentials in the cluster.
//                       A slot the exponentials kernel redid is skipped.
// A token's q-mass is exactly zero when its exponential is (a -inf draft logit, or one more
// than 87 T below the row maximum); q is out of mass once every token with mass has left.
#include "spec_verify.h"
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_dfwalk.cuh"
#include "sv_grid.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTrUnit = kTreeRefineUnit;  // logits per unit (one warp)
constexpr int kTrLane = kTrUnit / 32;     // logits per lane in a unit (contiguous)
constexpr int kRwThreads = 512;
constexpr int kRwWarps = kRwThreads / 32;
constexpr int kFinalChildren = 16;  // children of a reached node the grid-wide final re-draw replays
static_assert(kWarps >= kMaxTreeRefine, "one warp of the exponentials kernel per slot");

// The state of one slot's final re-draw at its reached node v, kept alike in every CTA:
// the implicit (p, q) of the re-walk (A, Dt, s in S_t units) and the pass in flight.
enum FinalState { kFinalNone = 0, kFinalAdvance = 1, kFinalPass = 2, kFinalDraw = 3 };
struct FinalSlot {
    df St, Sd, rho, A, Dt, s, erem;
    df Anext, s_new, total;  // the pending pass's coefficient and q scale; the draw's mass
    int seq, v, acc, nch, next, nrem, npos, npos_rem, state, ubuf;
    bool has_q, rejected, ready, add, lastpass;
};

// The listed sequences: the first kMaxTreeRefine with mark[b] != 0, in index order, into
// s_seq; returns how many are listed, *total = how many are marked.  Every CTA builds the
// same list.  s_bal: one word per warp of the CTA.
__device__ int list_marked(const int *mark, int B, int *s_seq, unsigned *s_bal, int *s_cnt, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) {
        s_cnt[0] = 0;
        s_cnt[1] = 0;
    }
    for (int base = 0; base < B; base += blockDim.x) {
        const int sq = base + tid;
        const int f = sq < B ? __ldcg(mark + sq) : 0;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, f != 0);
        if (lane == 0) s_bal[warp] = bal;
        __syncthreads();
        if (tid == 0) {
            for (int w = 0; w < nw; ++w) {
                unsigned m = s_bal[w];
                while (m) {
                    const int l = __ffs(m) - 1;
                    m &= m - 1;
                    if (s_cnt[0] < kMaxTreeRefine) s_seq[s_cnt[0]++] = base + w * 32 + l;
                    ++s_cnt[1];
                }
            }
        }
        __syncthreads();
    }
    *total = s_cnt[1];
    return s_cnt[0];
}

// The n-th marked sequence (0-based, index order), or -1 if fewer are marked; *total = how
// many are marked.  Every CTA computes the same.  s_bal: one word per warp of the CTA.
__device__ int nth_marked(const int *mark, int B, int n, unsigned *s_bal, int *s_cnt, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    if (tid == 0) {
        s_cnt[0] = -1;
        s_cnt[1] = 0;
    }
    for (int base = 0; base < B; base += blockDim.x) {
        const int sq = base + tid;
        const int f = sq < B ? __ldcg(mark + sq) : 0;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, f != 0);
        if (lane == 0) s_bal[warp] = bal;
        __syncthreads();
        if (tid == 0) {
            for (int w = 0; w < nw; ++w) {
                const unsigned m = s_bal[w];
                const int c = __popc(m);
                if (s_cnt[0] < 0 && n >= s_cnt[1] && n < s_cnt[1] + c) {
                    unsigned mm = m;
                    for (int q = 0; q < n - s_cnt[1]; ++q) mm &= mm - 1;
                    s_cnt[0] = base + w * 32 + __ffs(mm) - 1;
                }
                s_cnt[1] += c;
            }
        }
        __syncthreads();
    }
    *total = s_cnt[1];
    const int r = s_cnt[0];
    __syncthreads();  // read by every thread before the next call overwrites it
    return r;
}

// One unit of one row: e(j) = exp((x_j - M) / T) for its logits, stored; returns (to every
// lane) the unit sum, in lane order (lane sums, then a warp scan), and the number of
// positive e(j) in *cnt.
template <class D>
__device__ df exp_unit(const char *row, float M, df inv_t, int V, int u, df *E, int *cnt, int lane) {
    const int64_t j0 = int64_t(u) * kTrUnit + lane * kTrLane;
    df w[kDfLane];
    unit_exps<D>(row, M, inv_t, V, u, lane, w);  // 0 past the row's end
    int c = 0;
#pragma unroll
    for (int e = 0; e < kTrLane; ++e)
        if (j0 + e < V) {
            st_df(E + j0 + e, w[e]);
            c += df_pos(w[e]) ? 1 : 0;
        }
    *cnt = warp_reduce(c, [](int a, int b) { return a + b; });
    return unit_sum(w, lane);
}

// A sequence the walk marked only at its final draw, with the path recorded down to the
// node it reached (depth acc < K, acc + 1 records): its path is certain, so the re-walk
// starts at that node.
__device__ __forceinline__ bool final_only(int mark, int rlen, int acc, int K) {
    return mark == kTrMarkFinal && acc >= 0 && acc < K && rlen == acc + 1;
}

// The sums of the n stored values of a and of b (b may be null: 0) in warp_search's order --
// lane l adds its run [l per, (l + 1) per) in index order, then an inclusive scan over the
// lanes -- with each lane's loads of both lists in flight together.  Every lane returns
// both sums.
__device__ __forceinline__ void warp_totals2(const df *a, const df *b, int n, int lane, df *ta, df *tb) {
    constexpr int kB = 16;
    const int per = (n + 31) / 32;
    df sa = df_zero(), sb = df_zero();
    for (int q0 = 0; q0 < per; q0 += kB) {
        df va[kB], vb[kB];
#pragma unroll
        for (int q = 0; q < kB; ++q) {
            const int i = lane * per + q0 + q;
            const bool in = q0 + q < per && i < n;
            va[q] = in ? ldcg_df(a + i) : df_zero();
            vb[q] = (in && b) ? ldcg_df(b + i) : df_zero();
        }
#pragma unroll
        for (int q = 0; q < kB; ++q)
            if (q0 + q < per && lane * per + q0 + q < n) {
                sa = df_add(sa, va[q]);
                sb = df_add(sb, vb[q]);
            }
    }
    *ta = df_shfl(df_warp_scan(sa, lane), 31);
    *tb = df_shfl(df_warp_scan(sb, lane), 31);
}

// warp_search(vals, 1, n, 0, thr, false, ...) for n <= 32 kSearchRegs values, each lane's
// run loaded once (one round of loads; the crossing lane re-scans it from registers).
constexpr int kSearchRegs = 16;
__device__ __forceinline__ int search_regs(const df *vals, int n, df thr, df *run_out, bool *force_out, int lane) {
    const int per = (n + 31) / 32;
    df v[kSearchRegs];
#pragma unroll
    for (int q = 0; q < kSearchRegs; ++q) {
        const int i = lane * per + q;
        v[q] = (q < per && i < n) ? ldcg_df(vals + i) : df_zero();
    }
    df ls = df_zero();
    int lastpos = -1;
#pragma unroll
    for (int q = 0; q < kSearchRegs; ++q) {
        const int i = lane * per + q;
        if (q < per && i < n) {
            ls = df_add(ls, v[q]);
            if (df_pos(v[q])) lastpos = i;
        }
    }
    const df incl = df_warp_scan(ls, lane);
    df excl = df_shfl_up(incl, 1);
    if (lane == 0) excl = df_zero();
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, df_gt(df_add(df_zero(), incl), thr));
    if (bal) {
        const int l = __ffs(bal) - 1;
        int found = -1;
        df run = df_add(df_zero(), excl);
        if (lane == l) {
#pragma unroll
            for (int q = 0; q < kSearchRegs; ++q) {
                const int i = lane * per + q;
                if (found < 0 && q < per && i < n) {
                    const df nx = df_add(run, v[q]);
                    if (df_gt(nx, thr)) found = i;
                    else run = nx;
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
    *run_out = df_zero();
    *force_out = true;
    return warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
}

}  // namespace

// The exponentials of the recorded nodes of the first kMaxTreeRefine marked sequences
// (grid-stride over the (slot, position, row, unit) items that exist, one warp per unit,
// from the grid's last warp down), then the final re-draw of those marked only at their
// final draw by the first CTAs of the grid.
template <class D>
__global__ void __launch_bounds__(kThreads)
    tree_exp_kernel(Logits t, Logits d, int B, int N, int V, const int32_t *__restrict__ parent,
                    const int32_t *__restrict__ node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                    int without_replacement, int K, TreeRefineWs ws, int32_t *__restrict__ accepted_len,
                    int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_path) {
    __shared__ int s_seq[kMaxTreeRefine];
    __shared__ unsigned s_bal[kWarps];
    __shared__ int s_cnt[2];
    __shared__ FinalSlot s_fs[kMaxTreeRefine];
    __shared__ int s_fcn[kMaxTreeRefine][kFinalChildren], s_fcx[kMaxTreeRefine][kFinalChildren];
    __shared__ df s_fct[kMaxTreeRefine][kFinalChildren], s_fcd[kMaxTreeRefine][kFinalChildren];
    __shared__ int s_frt[kMaxTreeRefine][kFinalChildren];  // removed tokens and their coefficients
    __shared__ df s_frc[kMaxTreeRefine][kFinalChildren];
    __shared__ int s_fpt[kMaxTreeRefine][kTreeRecNodes];  // the path's tokens (the outputs before the final one)
    __shared__ int s_any;
    griddep_launch_next();
    griddep_wait();  // the walk's marks and records
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nunit = tree_refine_units(V);
    const df inv_t = df_div(df_from(1.f), df_from(T));
    const int64_t nw = int64_t(gridDim.x) * kWarps;
    const int64_t gw = int64_t(blockIdx.x) * kWarps + warp;
    int total = 0;
    const int n = list_marked(ws.mark, B, s_seq, s_bal, s_cnt, &total);
    if (blockIdx.x == 0 && threadIdx.x == 0) ws.ctl[kTrMarked] = total;
    if (n == 0) return;
    // the slots' records in shared memory (warp j, lane k): positions k0 .. k0 + nk - 1 have
    // exponentials to compute (a slot marked only at its final draw: the reached node alone)
    __shared__ float4 s_rec[kMaxTreeRefine][kTreeRecNodes];
    __shared__ int s_k0[kMaxTreeRefine], s_nk[kMaxTreeRefine], s_fo[kMaxTreeRefine];
    __shared__ int64_t s_ibase[kMaxTreeRefine + 1];
    if (warp < n) {
        const int64_t seq = s_seq[warp];
        const bool ok = SV_IN(seq, B);
        const int rlen = ok ? __ldcg(ws.rlen + seq) : 0;
        const int acc = ok ? __ldcg(accepted_len + seq) : -1;
        const bool fo = ok && final_only(__ldcg(ws.mark + seq), rlen, acc, K);
        const int rl = min(max(rlen, 0), min(K, kTreeRecNodes));
        if (lane < rl) s_rec[warp][lane] = __ldcg(ws.rec + seq * K + lane);
        if (lane == 0) {
            s_k0[warp] = fo ? acc : 0;
            s_nk[warp] = fo ? 1 : rl;
            s_fo[warp] = fo;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t b = 0;
        for (int jj = 0; jj < n; ++jj) {
            s_ibase[jj] = b;
            b += int64_t(s_nk[jj]) * 2 * nunit;
        }
        s_ibase[n] = b;
    }
    __syncthreads();
    const int64_t items = s_ibase[n];
    for (int64_t it = nw - 1 - gw; it < items; it += nw) {
        int j = 0;
        while (j + 1 < n && it >= s_ibase[j + 1]) ++j;
        const int64_t seq = s_seq[j];
        const int64_t loc = it - s_ibase[j];
        const int u = int(loc % nunit);
        const int r = int((loc / nunit) % 2);
        const int k = s_k0[j] + int(loc / (2 * int64_t(nunit)));
        if (!SV_IN(seq, B) || !SV_IN(k, kTreeRecNodes)) continue;
        const float4 rec = s_rec[j][k];
        const int node = __float_as_int(rec.x);
        if (r == 1 && rec.w == 0.f) continue;  // a leaf: no draft row
        const char *row = row_ptr(r == 0 ? t : d, D::kBytes, seq, node);
        const int64_t ek = (int64_t(j) * K + k) * 2 + r;
        int cnt = 0;
        const df us = exp_unit<D>(row, r == 0 ? rec.y : rec.z, inv_t, V, u, ws.et + ek * V, &cnt, lane);
        if (lane == 0) {
            st_df(ws.us + ek * nunit + u, us);
            if (r == 1 && cnt) atomicAdd(ws.npos + int64_t(j) * K + k, cnt);
        }
    }

    // ---- The final re-draw of the slots marked only at their final draw.  Every decision
    // on such a path was taken outside the fp32 error, so at the reached node v every child
    // was rejected (or v is a leaf): the rejections are replayed in double-float (each
    // child's test is taken again; one that now accepts leaves the slot to the re-walk),
    // each residual pass spread over the warps of the first P CTAs (one unit each), and the
    // final token drawn.  Those CTAs keep the same slot states: they change only through
    // sums of the same stored values in the same order.  Warp j owns slot j.  The other
    // CTAs only report their exponentials done at the first barrier.
    const int64_t pw = (int64_t(n) * nunit + kWarps - 1) / kWarps;
    const int P = pw < int64_t(gridDim.x) ? int(pw) : int(gridDim.x);
    if (int(blockIdx.x) >= P) {
        grid_arrive(ws.ctl);
        return;
    }
    if (warp < n) {
        FinalSlot &f = s_fs[warp];
        const int64_t seq = s_seq[warp];
        const bool fo = s_fo[warp];
        const int acc = fo ? s_k0[warp] : -1;
        const float4 rec = fo ? s_rec[warp][acc] : make_float4(0.f, 0.f, 0.f, 0.f);
        const int v = fo ? __float_as_int(rec.x) : -1;
        int nch = 0;  // v's children in index order (the walk tested them in this order)
        if (fo && v >= 0 && v < N)
            for (int base = v + 1; base < N; base += 32) {
                const int cn = base + lane;
                const bool ch = cn < N && __ldg(parent + cn) == v;
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, ch);
                const int idx = nch + __popc(bal & ((1u << lane) - 1u));
                if (ch && idx < kFinalChildren) s_fcn[warp][idx] = cn;
                nch += __popc(bal);
            }
        __syncwarp();
        const bool take = fo && v >= 0 && v < N && nch <= kFinalChildren;
        // the children's tokens and exponentials, as the exponentials above compute them
        if (take && lane < acc && SV_IN(lane + 1, kTreeRecNodes)) {  // the path below the root
            const int nx = __float_as_int(s_rec[warp][lane + 1].x);
            s_fpt[warp][lane] = SV_IN(nx, N) ? __ldg(node_tokens + seq * N + nx) : -1;
        }
        if (take && lane < nch) {
            const int cn = s_fcn[warp][lane];
            int x = __ldg(node_tokens + seq * N + cn);
            if (!SV_IN(x, V)) x = 0;  // (the walk checked the tokens before marking)
            s_fcx[warp][lane] = x;
            s_fct[warp][lane] = weight1_df(load_elem<D>(row_ptr(t, D::kBytes, seq, v), x), rec.y, inv_t);
            s_fcd[warp][lane] = weight1_df(load_elem<D>(row_ptr(d, D::kBytes, seq, v), x), rec.z, inv_t);
        }
        if (lane == 0) {
            f.seq = int(seq);
            f.v = v;
            f.acc = acc;
            f.nch = nch;
            f.state = take ? kFinalAdvance : kFinalNone;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int a = 0;
        for (int jj = 0; jj < n; ++jj) a |= s_fs[jj].state != kFinalNone;
        s_any = a;
    }
    __syncthreads();
    if (!s_any) return;  // (the same in every CTA of the P)
    if (!grid_barrier(ws.ctl)) return;  // every slot's exponentials, unit sums and support counts

    // The slot's stored rows at its reached node (position acc of the slot's records).
    auto rows_of = [&](int jj, const df **Et, const df **Ed, const df **Ut, const df **Ud) {
        const int64_t ek = (int64_t(jj) * K + s_fs[jj].acc) * 2;
        *Et = ws.et + ek * V;
        *Ed = *Et + V;
        *Ut = ws.us + ek * nunit;
        *Ud = *Ut + nunit;
    };
    if (warp < n && s_fs[warp].state == kFinalAdvance) {
        FinalSlot &f = s_fs[warp];
        const df *Et, *Ed, *Ut, *Ud;
        rows_of(warp, &Et, &Ed, &Ut, &Ud);
        const bool has_q = f.nch > 0;
        const int np = lane == 0 ? __ldcg(ws.npos + int64_t(warp) * K + f.acc) : 0;  // (in flight with the sums)
        df St, Sd;
        warp_totals2(Ut, has_q ? Ud : nullptr, nunit, lane, &St, &Sd);
        if (!has_q) Sd = df_from(1.f);
        if (lane == 0) {
            f.has_q = has_q;
            f.St = St;
            f.Sd = Sd;
            f.rho = has_q ? df_div(St, Sd) : df_zero();
            f.A = df_zero();
            f.Dt = St;
            f.s = df_from(1.f);
            f.erem = df_zero();
            f.npos = np;
            f.npos_rem = 0;
            f.nrem = 0;
            f.next = 0;
            f.rejected = false;
            f.ready = false;
        }
    }
    __syncthreads();

    // Slot j's next step (one thread): the next child's test; a rejection sets up the pass
    // under the new coefficient; after the last child the draw (a pass under the current
    // coefficients first when the last residual had no mass).
    auto advance = [&](int jj) {
        FinalSlot &f = s_fs[jj];
        if (f.next >= f.nch) {
            if (f.rejected && !f.ready) {
                f.Anext = f.A;
                f.add = false;
                f.lastpass = true;
                f.state = kFinalPass;
            } else {
                f.total = f.rejected ? f.Dt : f.St;
                f.state = kFinalDraw;
            }
            return;
        }
        const int c = f.next++;
        const int x = s_fcx[jj][c];
        const df ex_t = s_fct[jj][c], ex_d = s_fcd[jj][c];
        df ax = f.A;
        bool removed = false;
        for (int r = 0; r < f.nrem; ++r)
            if (s_frt[jj][r] == x) {
                ax = s_frc[jj][r];
                removed = true;
            }
        const df Wx = resid_w(ex_t, ex_d, df_mul(ax, f.rho));
        const float uu = uniform01(seed, offset, uint32_t(f.seq), uint32_t(s_fcn[jj][c] - 1), 0u);
        const df lhs = removed ? df_zero() : df_mul_f(df_mul(df_mul(f.s, ex_d), f.Dt), uu);
        if (df_lt(lhs, df_mul(Wx, f.Sd))) {  // accepted after all: the re-walk takes the slot
            f.state = kFinalNone;
            return;
        }
        f.rejected = true;
        const df Anew = df_add(f.A, df_mul(df_div(f.Dt, f.St), f.s));
        df s_new = f.s;
        const bool add = without_replacement && !removed;
        if (add) {
            if (SV_IN(f.nrem, kFinalChildren)) {
                s_frt[jj][f.nrem] = x;
                s_frc[jj][f.nrem] = Anew;
            }
            ++f.nrem;
            f.erem = df_add(f.erem, ex_d);
            if (df_pos(ex_d)) ++f.npos_rem;
            const df rest = df_sub(f.Sd, f.erem);
            s_new = (f.npos_rem >= f.npos || !df_pos(rest)) ? df_zero() : df_div(f.Sd, rest);
        }
        f.Anext = Anew;
        f.s_new = s_new;
        f.add = add;
        f.lastpass = false;
        f.state = kFinalPass;
    };
    // This lane's weights of unit u of slot jj under the coefficient a (removed tokens keep
    // theirs); e_t alone at a leaf.  0 past the row's end.
    auto unit_weights = [&](int jj, df a, const df *Et, const df *Ed, int u, df(&w)[kDfLane]) {
        const FinalSlot &f = s_fs[jj];
        const int64_t j0 = int64_t(u) * kTrUnit + lane * kTrLane;
        df xt[kTrLane], xd[kTrLane];  // the loads first, all in flight together
#pragma unroll
        for (int e = 0; e < kTrLane; ++e) {
            xt[e] = j0 + e < V ? ldcg_df(Et + j0 + e) : df_zero();
            xd[e] = (f.rejected && j0 + e < V) ? ldcg_df(Ed + j0 + e) : df_zero();
        }
        const df ar = df_mul(a, f.rho);
#pragma unroll
        for (int e = 0; e < kTrLane; ++e) {
            if (!f.rejected) {
                w[e] = xt[e];
                continue;
            }
            df arj = ar;
            for (int r = 0; r < f.nrem && r < kFinalChildren; ++r)
                if (s_frt[jj][r] == j0 + e) arj = df_mul(s_frc[jj][r], f.rho);
            w[e] = j0 + e < V ? resid_w(xt[e], xd[e], arj) : df_zero();
        }
    };

    for (int round = 0;; ++round) {
        if (lane == 0 && warp < n && s_fs[warp].state == kFinalAdvance) advance(warp);
        __syncthreads();
        bool any = false;
        for (int jj = 0; jj < n; ++jj) any |= s_fs[jj].state == kFinalPass;
        if (!any) break;  // (the same in every CTA)
        // the pass: (slot, unit) items over every warp of the grid, into buffer round & 1
        // (its readers of two rounds ago are past the barrier of the last round)
        df *umb = ws.um + int64_t(round & 1) * kMaxTreeRefine * nunit;
        for (int64_t it = gw; it < int64_t(n) * nunit; it += int64_t(P) * kWarps) {
            const int jj = int(it / nunit), u = int(it % nunit);
            if (s_fs[jj].state != kFinalPass) continue;  // (uniform over the warp)
            const df *Et, *Ed, *Ut, *Ud;
            rows_of(jj, &Et, &Ed, &Ut, &Ud);
            df w[kDfLane];
            unit_weights(jj, s_fs[jj].Anext, Et, Ed, u, w);
            const df us = unit_sum(w, lane);
            if (lane == 0) st_df(umb + int64_t(jj) * nunit + u, us);
        }
        if (!grid_barrier(ws.ctl, P)) return;
        if (warp < n && s_fs[warp].state == kFinalPass) {
            FinalSlot &f = s_fs[warp];
            df F, unused;
            warp_totals2(umb + int64_t(warp) * nunit, nullptr, nunit, lane, &F, &unused);
            if (lane == 0) {
                if (f.lastpass) {
                    f.total = F;
                    f.ubuf = round & 1;
                    f.state = kFinalDraw;
                } else {
                    if (df_pos(F)) {
                        f.A = f.Anext;
                        f.Dt = F;
                        f.ready = true;
                        f.ubuf = round & 1;
                    } else {  // no residual mass: p stays (the removal from q still happens)
                        f.ready = false;
                        if (f.add && SV_IN(f.nrem - 1, kFinalChildren)) s_frc[warp][f.nrem - 1] = f.A;
                    }
                    f.s = f.s_new;
                    f.state = kFinalAdvance;
                }
            }
        }
        __syncthreads();
    }

    // The draws (CTA 0, warp j for slot j): the unit holding u' x total by a prefix over the
    // unit masses in index order, then the logit inside it; the outputs rewritten.
    if (blockIdx.x != 0 || warp >= n || s_fs[warp].state != kFinalDraw) return;
    const FinalSlot &f = s_fs[warp];
    const df *Et, *Ed, *Ut, *Ud;
    rows_of(warp, &Et, &Ed, &Ut, &Ud);
    const df *umv = f.rejected ? ws.um + int64_t(f.ubuf) * kMaxTreeRefine * nunit + int64_t(warp) * nunit : Ut;
    const float u2 = uniform01(seed, offset, uint32_t(f.seq), uint32_t(f.v), 1u);
    const df thr = df_mul_f(f.total, u2);
    df run;
    bool force;
    int u = (nunit + 31) / 32 <= kSearchRegs ? search_regs(umv, nunit, thr, &run, &force, lane)
                                              : warp_search(umv, 1, nunit, df_zero(), thr, false, &run, &force, lane);
    if (u < 0) u = 0;
    if (u > nunit - 1) u = nunit - 1;
    df w[kDfLane];
    unit_weights(warp, f.A, Et, Ed, u, w);
    const int tok = unit_pick(w, int64_t(u) * kTrUnit, int64_t(u) * kTrUnit + lane * kTrLane, V, run, thr, force, lane);
    const int W = max_depth + 1;
    const int64_t sq = f.seq;
    int32_t *out = out_tokens + sq * W;
    int32_t *opath = out_path ? out_path + sq * W : nullptr;
    for (int i = lane; i < W; i += 32) {
        int o = -1, pth = -1;
        if (i <= f.acc && SV_IN(i, kTreeRecNodes)) pth = __float_as_int(s_rec[warp][i].x);
        if (i < f.acc && SV_IN(i, kTreeRecNodes)) o = s_fpt[warp][i];
        else if (i == f.acc) o = tok;
        out[i] = o;
        if (opath) opath[i] = pth;
    }
    if (lane == 0) {
        atomicOr(ws.ctl + kTrFinalDone, 1 << warp);
        atomicAdd(ws.ctl + kTrRedone, 1);
    }
}

// The re-walk: cluster j (CS CTAs) takes the marked sequences of rank j, j + 8, j + 16, ...
template <class D, int CS>
__global__ void __launch_bounds__(kRwThreads, 1)
    tree_rewalk_kernel(Logits t, Logits d, int B, int N, int V, const int32_t *__restrict__ parent,
                       const int32_t *__restrict__ node_tokens, int max_depth, float T, uint64_t seed,
                       uint64_t offset, int without_replacement, int K, TreeRefineWs ws,
                       int32_t *__restrict__ accepted_len, int32_t *__restrict__ out_tokens,
                       int32_t *__restrict__ out_path) {
    // shared: parent, token, child count [N]; removed tokens [N]; the CTA's removed tokens
    // [N]; path [max_depth + 1]; removed tokens' coefficients [N] and the CTA's x rho [N];
    // e_t and e_d at each child's token [N] (the current node's children)
    extern __shared__ int s_int[];
    int *s_par = s_int, *s_tok = s_int + N, *s_nch = s_int + 2 * N, *s_remtok = s_int + 3 * N;
    int *s_ltok = s_int + 4 * N, *s_path = s_int + 5 * N;
    df *s_remcoef = reinterpret_cast<df *>(s_int + 5 * N + max_depth + 1);
    df *s_lcoef = s_remcoef + N;
    df *s_cxt = s_lcoef + N, *s_cxd = s_cxt + N;
    __shared__ unsigned s_bal[kRwWarps];
    __shared__ int s_cnt[2];
    __shared__ df s_wsum[2][kRwWarps];
    __shared__ float s_wmax[2][kRwWarps];
    __shared__ int s_wcnt[kRwWarps];
    __shared__ df s_tot[2];
    __shared__ float s_max[2];
    __shared__ int s_ln, s_flag, s_tokout;
    griddep_launch_next();
    griddep_wait();  // the exponentials of the recorded nodes
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int j = int(blockIdx.x) / CS;
    const int rank = cluster_rank<CS>();
    const int nunit = tree_refine_units(V);
    auto unit_lo = [&](int c) { return int(int64_t(c) * nunit / CS); };
    const int u_lo = unit_lo(rank), u_hi = unit_lo(rank + 1);
    const int64_t e_lo = int64_t(u_lo) * kTrUnit, e_hi = int64_t(u_hi) * kTrUnit;
    const df inv_t = df_div(df_from(1.f), df_from(T));
    const int W = max_depth + 1;
    df *um = ws.um + int64_t(j) * nunit;            // unit masses of the current pass
    df *cpart = ws.part + int64_t(j) * 2 * CS * 2;  // [2 buffers][CS][2]
    float *cpmax = ws.pmax + int64_t(j) * CS * 2;
    int *ccnt = ws.pcnt + int64_t(j) * CS;

  // One marked sequence, walked again.  allow_cache: slot j holds its recorded rows'
  // exponentials (the first kMaxTreeRefine marked sequences); otherwise the cluster
  // computes every row's maxima and exponentials itself.
  auto walk_one = [&](int64_t seq, bool allow_cache) {
    int32_t *out = out_tokens + seq * W;
    int32_t *opath = out_path ? out_path + seq * W : nullptr;
    const int rlen = allow_cache ? __ldcg(ws.rlen + seq) : 0;

    // the tree (the walk checked it before marking the sequence)
    if (tid == 0) s_flag = 1;
    __syncthreads();
    for (int v = tid; v < N; v += kRwThreads) {
        const int p = parent[v];
        const int tk = v == 0 ? 0 : node_tokens[seq * N + v];
        s_par[v] = p;
        s_tok[v] = tk;
        s_nch[v] = 0;
        if ((v == 0 && p != -1) || (v > 0 && (p < 0 || p >= v)) || tk < 0 || tk >= V) s_flag = 0;
    }
    __syncthreads();
    if (!s_flag) return;  // (uniform over the cluster; never taken for a marked sequence)
    for (int v = 1 + tid; v < N; v += kRwThreads) atomicAdd(&s_nch[s_par[v]], 1);
    if (tid == 0) s_path[0] = 0;
    __syncthreads();

    auto fail = [&]() {
        if (rank != 0) return;
        for (int i = tid; i < W; i += kRwThreads) {
            out[i] = -1;
            if (opath) opath[i] = -1;
        }
        if (tid == 0) accepted_len[seq] = -1;
    };
    // The CTA's sums (warps in order) to cpart[buf][rank]; the cluster barrier; the
    // cluster's totals of both components (every thread, every CTA).
    // Both reductions are fixed butterflies in warp 0: lanes 0-15 take component 0, lanes
    // 16-31 component 1 (of warp `lane & 15`, then of CTA `lane & 15`, zeros past the end).
    static_assert(kRwWarps == 16 && CS <= 16, "half-warp butterflies");
    auto cluster_sums = [&](df a, df b, int buf, df *ta, df *tb) {
        if (lane == 0) {
            s_wsum[0][warp] = a;
            s_wsum[1][warp] = b;
        }
        __syncthreads();
        if (warp == 0) {
            df x = s_wsum[lane >> 4][lane & 15];
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) x = df_add(x, df_shfl_xor(x, o));
            if ((lane & 15) == 0) st_df(cpart + (buf * CS + rank) * 2 + (lane >> 4), x);
        }
        csync<CS>();
        if (warp == 0) {
            const int r = lane & 15;
            df x = r < CS ? ldcg_df(cpart + (buf * CS + r) * 2 + (lane >> 4)) : df_zero();
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) x = df_add(x, df_shfl_xor(x, o));
            if ((lane & 15) == 0) s_tot[lane >> 4] = x;
        }
        __syncthreads();
        *ta = s_tot[0];
        *tb = s_tot[1];
        __syncthreads();
    };

    // Marked only at its final draw, with the path recorded: start at the node the walk
    // reached (its path, every decision on it taken outside the fp32 error, is certain).
    int v = 0, depth = 0, buf = 0;
    {
        const int rl = __ldcg(ws.rlen + seq), acc = __ldcg(accepted_len + seq);
        if (final_only(__ldcg(ws.mark + seq), rl, acc, K)) {
            for (int i = tid; i <= acc; i += kRwThreads) s_path[i] = __float_as_int(__ldcg(ws.rec + seq * K + i).x);
            depth = acc;
            v = __float_as_int(__ldcg(ws.rec + seq * K + acc).x);
            if (!SV_IN(v, N)) v = 0, depth = 0;
            __syncthreads();
        }
    }
    for (;;) {
        const char *tp = row_ptr(t, D::kBytes, seq, v);
        const char *dp = row_ptr(d, D::kBytes, seq, v);
        const bool has_q = s_nch[v] > 0;
        // this depth's stored exponentials (a node deeper than K records reuses position
        // K - 1, whose node lies on the path above it and is no longer needed)
        const int pos = depth < K ? depth : K - 1;
        const int64_t ek = int64_t(j) * K + pos;
        const bool cached = depth < rlen && depth < K && __float_as_int(__ldcg(ws.rec + seq * K + depth).x) == v;
        df *Et = ws.et + ek * 2 * V, *Ed = Et + V;
        df *Ut = ws.us + ek * 2 * nunit, *Ud = Ut + nunit;
        int npos = 0;
        if (cached) {
            npos = __ldcg(ws.npos + ek);
        } else {
            // the rows' maxima, then their exponentials, in the cluster
            float mt = -__int_as_float(0x7f800000), md = -__int_as_float(0x7f800000);
            for (int u = u_lo + warp; u < u_hi; u += kRwWarps) {
                const int64_t j0 = int64_t(u) * kTrUnit + lane * kTrLane;
#pragma unroll
                for (int e = 0; e < kTrLane; ++e)
                    if (j0 + e < V) {
                        mt = max_nan(mt, load_elem<D>(tp, j0 + e));
                        if (has_q) md = max_nan(md, load_elem<D>(dp, j0 + e));
                    }
            }
            mt = warp_reduce(mt, [](float a, float b) { return max_nan(a, b); });
            md = warp_reduce(md, [](float a, float b) { return max_nan(a, b); });
            if (lane == 0) {
                s_wmax[0][warp] = mt;
                s_wmax[1][warp] = md;
            }
            __syncthreads();
            if (tid == 0) {
                float a = s_wmax[0][0], b = s_wmax[1][0];
                for (int w = 1; w < kRwWarps; ++w) {
                    a = max_nan(a, s_wmax[0][w]);
                    b = max_nan(b, s_wmax[1][w]);
                }
                cpmax[rank * 2] = a;
                cpmax[rank * 2 + 1] = b;
            }
            csync<CS>();
            if (tid == 0) {
                float a = __ldcg(cpmax), b = __ldcg(cpmax + 1);
                for (int c = 1; c < CS; ++c) {
                    a = max_nan(a, __ldcg(cpmax + c * 2));
                    b = max_nan(b, __ldcg(cpmax + c * 2 + 1));
                }
                s_max[0] = a;
                s_max[1] = b;
            }
            __syncthreads();
            const float Mt = s_max[0], Md = s_max[1];
            csync<CS>();  // every CTA has read cpmax before it can be written again
            if (!is_finite(Mt) || (has_q && !is_finite(Md))) {  // not a distribution (R11)
                fail();
                return;
            }
            int cnt = 0;
            for (int u = u_lo + warp; u < u_hi; u += kRwWarps) {
                int c0 = 0, c1 = 0;
                const df a = exp_unit<D>(tp, Mt, inv_t, V, u, Et, &c0, lane);
                if (lane == 0) st_df(Ut + u, a);
                if (has_q) {
                    const df b = exp_unit<D>(dp, Md, inv_t, V, u, Ed, &c1, lane);
                    if (lane == 0) st_df(Ud + u, b);
                    cnt += c1;
                }
            }
            if (lane == 0) s_wcnt[warp] = cnt;
            __syncthreads();
            if (tid == 0) {
                int m = 0;
                for (int w = 0; w < kRwWarps; ++w) m += s_wcnt[w];
                ccnt[rank] = m;
            }
            csync<CS>();
            if (tid == 0) {
                int m = 0;
                for (int c = 0; c < CS; ++c) m += __ldcg(ccnt + c);
                s_wcnt[0] = m;
            }
            __syncthreads();
            npos = s_wcnt[0];
            csync<CS>();  // every CTA has read ccnt
        }
        // the rows' sums from the unit sums: each warp its units u_lo + warp + 16 i (lane i;
        // a loop for runs of more than 512 units), a butterfly, then the cluster's reduction
        df ct = df_zero(), cd = df_zero();
        for (int u0 = u_lo + warp; u0 < u_hi; u0 += kRwWarps * 32) {
            const int u = u0 + kRwWarps * lane;
            df a = u < u_hi ? ldcg_df(Ut + u) : df_zero();
            df b = (has_q && u < u_hi) ? ldcg_df(Ud + u) : df_zero();
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a = df_add(a, df_shfl_xor(a, o));
                b = df_add(b, df_shfl_xor(b, o));
            }
            ct = df_add(ct, a);
            cd = df_add(cd, b);
        }
        df St, Sd;
        cluster_sums(ct, cd, buf, &St, &Sd);
        if (!has_q) Sd = df_from(1.f);
        int dbuf = buf;  // the buffer the final draw reads (e_t's sums at a leaf)
        buf ^= 1;
        const df rho = has_q ? df_div(St, Sd) : df_zero();
        df *umv = Ut;  // the unit masses the final draw reads
        for (int cn = v + 1 + tid; cn < N; cn += kRwThreads)  // the children's e_t, e_d, loaded together
            if (s_par[cn] == v) {
                s_cxt[cn] = ldcg_df(Et + s_tok[cn]);
                s_cxd[cn] = ldcg_df(Ed + s_tok[cn]);
            }
        __syncthreads();

        // One residual pass under coefficient a (removed tokens keep theirs): unit masses
        // and the cluster's total.
        int nrem = 0;
        auto mass_pass = [&](df a) -> df {
            const df ar = df_mul(a, rho);
            if (tid == 0) {
                int m = 0;
                for (int r = 0; r < nrem; ++r)
                    if (s_remtok[r] >= e_lo && s_remtok[r] < e_hi) {
                        s_ltok[m] = s_remtok[r];
                        s_lcoef[m] = df_mul(s_remcoef[r], rho);
                        ++m;
                    }
                s_ln = m;
            }
            __syncthreads();
            const int ln = s_ln;
            df cw = df_zero();
            for (int u = u_lo + warp; u < u_hi; u += kRwWarps) {
                const int64_t j0 = int64_t(u) * kTrUnit + lane * kTrLane;
                df xt[kTrLane], xd[kTrLane];  // the loads first, all in flight together
#pragma unroll
                for (int e = 0; e < kTrLane; ++e) {
                    xt[e] = j0 + e < V ? ldcg_df(Et + j0 + e) : df_zero();
                    xd[e] = j0 + e < V ? ldcg_df(Ed + j0 + e) : df_zero();
                }
                DfSum ls;
#pragma unroll
                for (int e = 0; e < kTrLane; ++e)
                    if (j0 + e < V) {
                        df arj = ar;
                        for (int q = 0; q < ln; ++q)
                            if (s_ltok[q] == j0 + e) arj = s_lcoef[q];
                        ls.add(resid_w(xt[e], xd[e], arj));
                    }
                const df us = df_shfl(df_warp_scan(ls.value(), lane), 31);
                if (lane == 0) {
                    st_df(um + u, us);
                    cw = df_add(cw, us);
                }
            }
            df tot, unused;
            cluster_sums(cw, df_zero(), buf, &tot, &unused);
            dbuf = buf;
            buf ^= 1;
            umv = um;
            return tot;
        };

        // the children in order, against the implicit (p, q): p(x) = W(x) / Dt,
        // q(x) = s e_d(x) / S_d (0 once removed)
        df A = df_zero(), Dt = St, s = df_from(1.f), erem = df_zero();
        int npos_rem = 0, next = -1;
        bool rejected = false, ready = false;
        for (int cn = v + 1; cn < N && next < 0; ++cn) {
            if (s_par[cn] != v) continue;
            const int x = s_tok[cn];
            const df ex_t = s_cxt[cn], ex_d = s_cxd[cn];
            df ax = A;
            bool removed = false;
            for (int r = 0; r < nrem; ++r)
                if (s_remtok[r] == x) {
                    ax = s_remcoef[r];
                    removed = true;
                }
            const df Wx = resid_w(ex_t, ex_d, df_mul(ax, rho));
            const float uu = uniform01(seed, offset, uint32_t(seq), uint32_t(cn - 1), 0u);
            // u q(x) < p(x)  <=>  u s e_d(x) Dt < W(x) S_d  (both sides cleared of divisions)
            const df lhs = removed ? df_zero() : df_mul_f(df_mul(df_mul(s, ex_d), Dt), uu);
            if (df_lt(lhs, df_mul(Wx, Sd))) {
                next = cn;
                break;
            }
            rejected = true;
            const df Anew = df_add(A, df_mul(df_div(Dt, St), s));
            df s_new = s;
            const bool add = without_replacement && !removed;
            if (add) {
                if (tid == 0 && SV_IN(nrem, N)) {
                    s_remtok[nrem] = x;
                    s_remcoef[nrem] = Anew;
                }
                ++nrem;
                erem = df_add(erem, ex_d);
                if (df_pos(ex_d)) ++npos_rem;
                const df rest = df_sub(Sd, erem);
                s_new = (npos_rem >= npos || !df_pos(rest)) ? df_zero() : df_div(Sd, rest);
            }
            __syncthreads();
            const df F = mass_pass(Anew);
            if (df_pos(F)) {
                A = Anew;
                Dt = F;
                ready = true;
            } else {  // no residual mass: p stays (the removal from q still happens)
                ready = false;
                if (add && tid == 0) s_remcoef[nrem - 1] = A;
            }
            s = s_new;
            __syncthreads();
        }
        if (next >= 0) {
            ++depth;
            if (tid == 0 && depth <= max_depth && SV_IN(next, N)) s_path[depth] = next;
            __syncthreads();
            if (depth > max_depth) {  // (the walk checked the depths; never taken)
                fail();
                return;
            }
            v = next;
            continue;
        }
        // the final token at v: e_t at a leaf, else the last residual (or, when the last
        // one had no mass, the weights under the current coefficients)
        df total = St;
        if (rejected) total = ready ? Dt : mass_pass(A);
        if (rank != 0) return;
        if (warp == 0) {
            const float u2 = uniform01(seed, offset, uint32_t(seq), uint32_t(v), 1u);
            const df thr = df_mul_f(total, u2);
            df run;
            bool force;
            int c = warp_search(cpart + dbuf * CS * 2, 2, CS, df_zero(), thr, false, &run, &force, lane);
            if (c < 0) c = 0;
            const int clo = unit_lo(c), chi = unit_lo(c + 1);
            int u = warp_search(umv + clo, 1, chi - clo, run, thr, force, &run, &force, lane);
            u = clo + (u < 0 ? 0 : u);
            if (u > nunit - 1) u = nunit - 1;
            // inside the unit: the same weights and order as the pass that summed it
            const df arA = df_mul(A, rho);
            const int64_t j0 = int64_t(u) * kTrUnit + lane * kTrLane;
            df w[kTrLane];
            DfSum lsum;
            int lastpos = -1;
#pragma unroll
            for (int e = 0; e < kTrLane; ++e) {
                w[e] = df_zero();
                if (j0 + e < V) {
                    if (!rejected) {
                        w[e] = ldcg_df(Et + j0 + e);
                    } else {
                        df arj = arA;
                        for (int r = 0; r < nrem; ++r)
                            if (s_remtok[r] == j0 + e) arj = df_mul(s_remcoef[r], rho);
                        w[e] = resid_w(ldcg_df(Et + j0 + e), ldcg_df(Ed + j0 + e), arj);
                    }
                    lsum.add(w[e]);
                    if (df_pos(w[e])) lastpos = int(j0) + e;
                }
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
                    // the lane's own logits in order; rounding past its end: its last positive one
                    int cand = -1, lpos = -1;
                    df r2 = df_add(run, excl);
#pragma unroll
                    for (int e = 0; e < kTrLane; ++e) {
                        const df nx = df_add(r2, w[e]);
                        if (cand < 0 && df_gt(nx, thr)) cand = int(j0) + e;
                        if (df_pos(w[e])) lpos = int(j0) + e;
                        r2 = nx;
                    }
                    if (cand < 0) cand = lpos;
                    cand = __shfl_sync(0xFFFFFFFFu, cand, l);
                    if (cand >= 0) tok = cand;
                }
            }
            if (tok < 0) tok = int(int64_t(u) * kTrUnit);
            if (lane == 0) s_tokout = tok;
        }
        __syncthreads();
        const int tok = s_tokout;
        for (int i = tid; i < W; i += kRwThreads) {
            int o = -1, pth = -1;
            if (i <= depth) pth = s_path[i];
            if (i < depth) o = SV_IN(s_path[i + 1], N) ? s_tok[s_path[i + 1]] : -1;
            else if (i == depth) o = tok;
            out[i] = o;
            if (opath) opath[i] = pth;
        }
        if (tid == 0) accepted_len[seq] = depth;
        return;
    }
  };

    // nothing left: every marked sequence was a slot the exponentials kernel re-drew (the
    // same words in every CTA)
    if (__ldcg(ws.ctl + kTrMarked) == __popc(__ldcg(ws.ctl + kTrFinalDone))) return;
    // cluster j takes the marked sequences of rank j, j + G, j + 2 G, ... (index order; G
    // clusters), the first of them with slot j's stored exponentials
    const int G = int(gridDim.x) / CS;
    for (int iter = 0;; ++iter) {
        int total_marked = 0;
        const int64_t seq = nth_marked(ws.mark, B, j + iter * G, s_bal, s_cnt, &total_marked);
        if (seq < 0 || !SV_IN(seq, B)) break;  // (the whole cluster)
        // a slot the exponentials kernel re-drew (the same word in every CTA)
        if (iter == 0 && ((__ldcg(ws.ctl + kTrFinalDone) >> j) & 1)) continue;
        walk_one(seq, iter == 0);
        csync<CS>();  // every CTA is done with the slot's scratch before the next sequence
        if (rank == 0 && tid == 0) atomicAdd(ws.ctl + kTrRedone, 1);
    }
}

cudaError_t launch_tree_exp(int dtype, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                            const int32_t *node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                            int without_replacement, int K, TreeRefineWs ws, int32_t *accepted_len,
                            int32_t *out_tokens, int32_t *out_path, cudaStream_t s) {
    auto ke = dtype == 1 ? tree_exp_kernel<BF16> : tree_exp_kernel<F32>;
    unsigned grid = 0;  // every resident CTA (a cooperative launch: its passes meet at grid barriers)
    cudaError_t e = persistent_grid(ke, int64_t(1) << 40, &grid);
    if (e == cudaSuccess)
        e = launch_after_ex(true, ke, grid, kThreads, 0, s, t, d, B, N, V, parent, node_tokens, max_depth, T, seed,
                            offset, without_replacement, K, ws, accepted_len, out_tokens, out_path);
    return e;
}

namespace {
template <int CS>
cudaError_t launch_rewalk(int dtype, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                          const int32_t *node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                          int without_replacement, int K, TreeRefineWs ws, int32_t *accepted_len, int32_t *out_tokens,
                          int32_t *out_path, cudaStream_t s, bool probe, int *fits) {
    auto kw = dtype == 1 ? tree_rewalk_kernel<BF16, CS> : tree_rewalk_kernel<F32, CS>;
    const size_t smem = tree_refine_smem(N, max_depth);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) e = cudaFuncSetAttribute(kw, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess && CS > 8) e = cudaFuncSetAttribute(kw, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(kMaxTreeRefine * CS));
    cfg.blockDim = dim3(kRwThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (probe) {  // can a cluster of this size be resident at all?
        cfg.numAttrs = 1;
        return cudaOccupancyMaxActiveClusters(fits, kw, &cfg);
    }
    return cudaLaunchKernelEx(&cfg, kw, t, d, B, N, V, parent, node_tokens, max_depth, T, seed, offset,
                              without_replacement, K, ws, accepted_len, out_tokens, out_path);
}
}  // namespace

// Clusters of 16 CTAs where the device can hold one (a non-portable size), else of 8.
cudaError_t launch_tree_rewalk(int dtype, Logits t, Logits d, int B, int N, int V, const int32_t *parent,
                               const int32_t *node_tokens, int max_depth, float T, uint64_t seed, uint64_t offset,
                               int without_replacement, int K, TreeRefineWs ws, int32_t *accepted_len,
                               int32_t *out_tokens, int32_t *out_path, cudaStream_t s) {
    static_assert(kTreeRefineCluster == 16, "the per-sequence scratch is sized for clusters of up to 16");
    int fits = 0;
    cudaError_t e = launch_rewalk<16>(dtype, t, d, B, N, V, parent, node_tokens, max_depth, T, seed, offset,
                                      without_replacement, K, ws, accepted_len, out_tokens, out_path, s, true, &fits);
    if (e == cudaSuccess && fits >= 1)
        return launch_rewalk<16>(dtype, t, d, B, N, V, parent, node_tokens, max_depth, T, seed, offset,
                                 without_replacement, K, ws, accepted_len, out_tokens, out_path, s, false, nullptr);
    (void)cudaGetLastError();  // a refused size is not an error of this call
    return launch_rewalk<8>(dtype, t, d, B, N, V, parent, node_tokens, max_depth, T, seed, offset,
                            without_replacement, K, ws, accepted_len, out_tokens, out_path, s, false, nullptr);
}

}  // namespace sv
