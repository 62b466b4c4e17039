// sv_typical.cu -- verification rules that read target rows only, lazily, one CTA per
// sequence: typical acceptance (Medusa's relaxed rule) and sampling verification against a
// one-hot draft distribution (the prompt-lookup drafter's q).
//
// Method ("7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead", the Medusa
// paragraph and the closing note on typical acceptance): a draft token is accepted when its
// target probability exceeds a threshold that scales with the step's entropy; the rule
// does not preserve the target law.  The form taken (the pages give no constants):
// tau_i = min(epsilon, delta exp(-H(p_i))) with p_i = softmax(t_i / T); the first draft with
// p_i(x_i) <= tau_i ends the prefix and the token at the stop is drawn from p itself.
//
// With a one-hot q (q_i(x_i) = 1) the chain rule of "The rule" becomes: accept x_i iff
// u_i < p_i(x_i) (u_i = U(b, i, purpose 0)); at the first rejection k the residual
// (p_k - q_k)+ is p_k with x_k removed, so the final token is drawn from p_k without x_k;
// the bonus at k = gamma from p_gamma.  No draft logits exist or are read.
//
// The rule needs rows 0 .. k only.  Per row read, one pass gives (M, S, Z): the maximum,
// S = sum 2^a and Z = sum 2^a a with a = (x - M) log2(e) / T, merged across units with the
// usual rescaling (Z of a part relative to the new maximum is 2^d (Z + d S), d = the
// shift); then p(x) = 2^a(x) / S and H = ln S - ln 2 Z / S.  At the stop row a second pass
// stores the unit masses of p and the final token is drawn as in the tree walk: double-float
// prefixes over the units, the lane whose run crosses u' x total, then one logit per lane.
#include "sv_device.cuh"
#include "sv_df.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kTyThreads = 1024;
constexpr int kTyWarps = kTyThreads / 32;

struct Stat3 {
    float M, S, Z;  // max; sum of 2^a; sum of 2^a a (a in log2 units, relative to M)
};

__device__ __forceinline__ void add_part(Stat3 &r, const Stat3 &p, float c) {
    if (!(p.S > 0.f)) return;  // an empty or all -inf part
    const float d = __fmul_rn(__fsub_rn(p.M, r.M), c);  // <= 0
    const float f = ex2(d);
    r.S = fmaf(p.S, f, r.S);
    r.Z = fmaf(f, fmaf(d, p.S, p.Z), r.Z);
}
// p's weight 2^((x - M) c) / S for the draw, with c = c_hi + c_lo (log2(e) / T to ~48 bits)
// and the product's rounding error carried as a first-order correction: 2^(a + r) =
// 2^a (1 + r ln 2) to ~1e-14.  Without it the fp32 rounding of c and of the argument shifts
// every weight by ~6e-8 |a| -- the same way for all of them, so prefix sums drift by
// ~1e-7 of the total, more than a draw near a CDF boundary can absorb.
__device__ __forceinline__ float pweight(float x, float M, float c_hi, float c_lo, float inv_s) {
    const float xm = __fsub_rn(x, M);
    if (!(xm > -__int_as_float(0x7f800000))) return 0.f;  // a -inf logit
    const float a = __fmul_rn(xm, c_hi);
    const float r = __fadd_rn(__fmaf_rn(xm, c_hi, -a), __fmul_rn(xm, c_lo));
    const float e = ex2(a);
    return __fmul_rn(__fmaf_rn(e, __fmul_rn(r, 0.69314718f), e), inv_s);
}

// (M, S, Z) of the union of two parts; a NaN or +inf maximum makes the result invalid.
__device__ __forceinline__ Stat3 merge3(const Stat3 &a, const Stat3 &b, float c) {
    Stat3 r{max_nan(a.M, b.M), 0.f, 0.f};
    if (!is_finite(r.M)) return r;
    add_part(r, a, c);
    add_part(r, b, c);
    return r;
}

}  // namespace

template <class D, bool VEC>
__global__ void __launch_bounds__(kTyThreads, 1)
    typical_walk_kernel(Logits t, int gamma, int V, const int32_t *__restrict__ tokens, float c, float c_lo,
                        int onehot, float epsilon, float delta, uint64_t seed, uint64_t offset, int nunit,
                        float *umass, TreeRefineWs rw,
                        int32_t *__restrict__ accepted_len, int32_t *__restrict__ out_tokens) {
    __shared__ Stat3 s_st[kTyWarps];
    __shared__ Stat3 s_row;
    __shared__ int s_flag, s_tok, s_near;
    griddep_launch_next();
    griddep_wait();  // the caller's kernels may still be writing the inputs
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t seq = blockIdx.x;
    const int G1 = gamma + 1;
    int32_t *out = out_tokens + seq * G1;
    const int32_t *x = tokens + seq * gamma;
    float *um = umass + seq * int64_t(nunit);
    constexpr int RE = res_tile_elems<D>();

    if (blockIdx.x == 0) {  // the re-draw's control words and counters (it starts after this grid)
        if (tid < kTrCtlWords) rw.ctl[tid] = 0;
        if (tid < kMaxTreeRefine) rw.npos[tid] = 0;
    }
    if (tid == 0) {
        s_flag = 1;
        s_near = 0;
    }
    __syncthreads();
    for (int i = tid; i < gamma; i += kTyThreads)
        if (x[i] < 0 || x[i] >= V) s_flag = 0;
    __syncthreads();
    auto fail = [&]() {
        for (int i = tid; i < G1; i += kTyThreads) out[i] = -1;
        if (tid == 0) {
            accepted_len[seq] = -1;
            rw.mark[seq] = 0;
            rw.rlen[seq] = 0;
        }
    };
    if (!s_flag) {
        fail();
        return;
    }

    // (M, S, Z) of one row: warps over units (lane l holds vectors l, l + 32, ...), a fixed
    // merge order within a warp and across warps; every thread returns the row's result.
    auto row_stats = [&](const char *row) -> Stat3 {
        Stat3 ws{-__int_as_float(0x7f800000), 0.f, 0.f};
        for (int u = warp; u < nunit; u += kTyWarps) {
            const int64_t u0 = int64_t(u) * RE;
            const int len = unit_len(V, u0, RE);
            uint4 v[kResVecs];
#pragma unroll
            for (int k = 0; k < kResVecs; ++k) {
                const int e0 = (lane + 32 * k) * D::EPV;
                v[k] = e0 < len ? load_vec<D, VEC>(row, u0, e0, len) : neg_inf_vec<D>();
            }
            const float m = warp_reduce(thread_max<D>(v), [](float a, float b) { return max_nan(a, b); });
            float sv = 0.f, zv = 0.f;
            if (is_finite(m)) {
#pragma unroll
                for (int k = 0; k < kResVecs; ++k)
#pragma unroll
                    for (int e = 0; e < D::EPV; ++e) {
                        const float a = __fmul_rn(__fsub_rn(vec_elem<D>(v[k], e), m), c);
                        const float w = ex2(a);  // 0 for a -inf logit
                        sv += w;
                        zv += w > 0.f ? w * a : 0.f;
                    }
            }
            sv = warp_reduce(sv, [](float a, float b) { return a + b; });
            zv = warp_reduce(zv, [](float a, float b) { return a + b; });
            ws = merge3(ws, Stat3{m, sv, zv}, c);
        }
        if (lane == 0) s_st[warp] = ws;
        __syncthreads();
        if (tid == 0) {
            Stat3 r = s_st[0];
            for (int w = 1; w < kTyWarps; ++w) r = merge3(r, s_st[w], c);
            s_row = r;
        }
        __syncthreads();
        const Stat3 r = s_row;
        __syncthreads();
        return r;
    };

    int k = gamma;
    Stat3 st{};
    for (int i = 0; i <= gamma; ++i) {
        const char *row = row_ptr(t, D::kBytes, seq, i);
        st = row_stats(row);
        if (!is_finite(st.M) || !(st.S > 0.f)) {  // not a distribution (R11)
            fail();
            return;
        }
        if (i == gamma) break;
        const float px = __fdiv_rn(ex2(__fmul_rn(__fsub_rn(load_elem<D>(row, x[i]), st.M), c)), st.S);
        bool accept;
        if (onehot) {  // u q(x) < p(x) with q(x) = 1
            accept = uniform01(seed, offset, uint32_t(seq), uint32_t(i), 0u) < px;
        } else {
            const float H = __fsub_rn(logf(st.S), __fdiv_rn(0.69314718f * st.Z, st.S));
            accept = px > fminf(epsilon, delta * expf(-H));
        }
        if (!accept) {
            k = i;
            break;
        }
    }
    // one-hot q after a rejection: the residual is p_k without the rejected token
    const int xk = (onehot && k < gamma) ? x[k] : -1;

    // the final token from p_k: unit masses, then the draw
    const char *row = row_ptr(t, D::kBytes, seq, k);
    const float inv_s = 1.f / st.S;
    for (int u = warp; u < nunit; u += kTyWarps) {
        const int64_t u0 = int64_t(u) * RE;
        const int len = unit_len(V, u0, RE);
        uint4 v[kResVecs];
#pragma unroll
        for (int q = 0; q < kResVecs; ++q) {
            const int e0 = (lane + 32 * q) * D::EPV;
            v[q] = e0 < len ? load_vec<D, VEC>(row, u0, e0, len) : neg_inf_vec<D>();
        }
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < kResVecs; ++q)
#pragma unroll
            for (int e = 0; e < D::EPV; ++e) {
                const int j = int(u0) + (lane + 32 * q) * D::EPV + e;
                acc += j == xk ? 0.f : pweight(vec_elem<D>(v[q], e), st.M, c, c_lo, inv_s);
            }
        acc = warp_reduce(acc, [](float a, float b) { return a + b; });
        if (lane == 0) um[u] = acc;
    }
    __syncthreads();  // the unit masses of every warp (global, this CTA's own)
    if (warp == 0) {
        const float u2 = uniform01(seed, offset, uint32_t(seq), uint32_t(k), 1u);
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
        constexpr int NE = kResVecs * D::EPV;  // logits per lane
        const int64_t u0 = int64_t(unit) * RE;
        const int len = unit_len(V, u0, RE);
        PairSum lsum;
        int lastpos = -1;
#pragma unroll
        for (int q = 0; q < kResVecs; ++q) {
            const int e0 = (lane * kResVecs + q) * D::EPV;
            const uint4 vv = e0 < len ? load_vec<D, VEC>(row, u0, e0, len) : neg_inf_vec<D>();
#pragma unroll
            for (int e = 0; e < D::EPV; ++e) {
                const float w = int(u0) + e0 + e == xk ? 0.f : pweight(vec_elem<D>(vv, e), st.M, c, c_lo, inv_s);
                lsum.add(w);
                if (e0 + e < len && w > 0.f) lastpos = e0 + e;
            }
        }
        const df lincl = df_warp_scan(lsum.value(), lane);
        df lexcl = df_shfl_up(lincl, 1);
        if (lane == 0) lexcl = df{0.f, 0.f};
        int first = -1;
        float gap = 0.f;  // distance of thr to the chosen token's CDF boundaries
        const unsigned lb = force_last ? 0u : __ballot_sync(0xFFFFFFFFu, df_gt(df_add(base, lincl), thr));
        if (lb) {
            const int l3 = __ffs(lb) - 1;
            const int j = l3 * NE + lane;
            const float w = (lane < NE && j < len && int(u0) + j != xk)
                                ? pweight(load_elem<D>(row, u0 + j), st.M, c, c_lo, inv_s)
                                : 0.f;
            const df start = df_add(base, df_shfl(lexcl, l3));
            const df above = df_sub(df_add(start, df_warp_scan(df_from(w), lane)), thr);
            const unsigned eb = __ballot_sync(0xFFFFFFFFu, lane < NE && j < len && df_pos(above));
            if (eb) {
                const int le = __ffs(eb) - 1;
                first = l3 * NE + le;
                const float ah = __shfl_sync(0xFFFFFFFFu, above.hi, le);
                const float wl = __shfl_sync(0xFFFFFFFFu, w, le);
                gap = fminf(__fsub_rn(wl, ah), ah);  // thr - C_{j-1} = w - (C_j - thr)
            }
        }
        // fp32 weights (~1e-7 each) cannot settle a threshold this close: the double-float
        // re-draw redoes it
        if (lane == 0 && (first < 0 || force_last || !(gap >= kTypicalCdfWindow * totd.hi + token_window(st.S))))
            s_near = 1;
        lastpos = warp_reduce(lastpos, [](int a, int b) { return max(a, b); });
        int tok = first >= 0 ? first : lastpos;
        if (tok < 0) tok = 0;
        if (lane == 0) s_tok = int(u0) + tok;
    }
    __syncthreads();
    for (int i = tid; i < G1; i += kTyThreads) out[i] = i < k ? x[i] : (i == k ? s_tok : -1);
    if (tid == 0) {
        accepted_len[seq] = k;
        rw.mark[seq] = s_near;
        rw.rlen[seq] = 1;  // the stop row and its maximum, for the re-draw
        rw.rec[seq] = make_float4(__int_as_float(k), st.M, __int_as_float(xk), 0.f);  // .z: the excluded token
    }
}

cudaError_t launch_typical(int dtype, bool vec, Logits t, int B, int gamma, int V, const int32_t *tokens, float c,
                           float c_lo, int onehot, float epsilon, float delta, uint64_t seed, uint64_t offset,
                           int nunit, float *umass, TreeRefineWs rw, int32_t *accepted_len, int32_t *out_tokens,
                           cudaStream_t s) {
    auto k = dtype == 1 ? (vec ? typical_walk_kernel<BF16, true> : typical_walk_kernel<BF16, false>)
                        : (vec ? typical_walk_kernel<F32, true> : typical_walk_kernel<F32, false>);
    return launch_after(k, unsigned(B), kTyThreads, 0, s, t, gamma, V, tokens, c, c_lo, onehot, epsilon, delta, seed,
                        offset,
                        nunit, umass, rw, accepted_len, out_tokens);
}

}  // namespace sv
