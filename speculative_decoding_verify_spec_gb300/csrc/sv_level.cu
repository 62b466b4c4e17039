// sv_level.cu -- level-synchronous LAZY verification of the rules that walk the target rows
// left to right: the sampling chain (accept x_i with probability min(1, p(x)/q(x))), sampling
// against a one-hot draft distribution (accept iff u < p(x)), and typical acceptance (accept
// iff p(x) > min(epsilon, delta e^-H)).
//
// Method ("7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead", "Extending to
// a chain of gamma draft tokens": the first rejection ends the round, so the rows after it
// never reach the result; "Rollback": only the accepted prefix is kept).  The rows a
// sequence needs are rows 0 .. k of its own stop k, so they are read level by level: at
// level i every sequence still walking streams its target row i (and draft row i), over the
// whole GPU, 4 KB tile by 4 KB tile, with the row-statistics kernel's per-tile arithmetic.
// Each CTA takes a contiguous range of the level's tiles and, once its range is done, adds
// its tile count to a counter per sequence it touched; the CTA that completes a sequence's
// count merges the tile partials in the fixed order the eager decide uses, takes that
// level's accept test, and either stops the sequence -- writing its plan (stop row, kind of
// draw), its accepted prefix and the -1 padding, exactly as decide does -- or lists it for
// the next level.  A grid barrier ends each level (the launch is cooperative), and the walk
// ends at the first level nobody reaches.  The residual masses, the draw and the double-float
// re-draw of near-boundary sequences are then the eager path's own kernels on the plans,
// statistics and tile partials written here: for the chain rule the lazy result is the eager
// one bit for bit whenever every row is a distribution.
//
// A sequence whose accept test came near its threshold (marked for the double-float rescan)
// keeps streaming every later row, so the rescan finds whichever stop the exact test gives;
// the rows it could use are counted in lavail.
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_grid.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kLvThreads = 768;  // one CTA per SM (fewer CTAs meet at each barrier), 84 registers a thread

// (M, S, Z) of a set of logits: the maximum, S = sum 2^a and Z = sum 2^a a with
// a = (x - M) c (base-2 units relative to M).  Merging moves a part to a new maximum with
// d = (M_part - M) c <= 0:  S <- 2^d S,  Z <- 2^d (Z + d S).
struct Stat3 {
    float M, S, Z;
};
__device__ __forceinline__ Stat3 merge3(Stat3 a, Stat3 b, float c) {
    Stat3 r{max_nan(a.M, b.M), 0.f, 0.f};
    if (!is_finite(r.M)) return r;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const Stat3 p = k == 0 ? a : b;
        if (!(p.S > 0.f)) continue;  // an empty or all -inf part
        const float dd = __fmul_rn(__fsub_rn(p.M, r.M), c);
        const float f = ex2(dd);
        r.S = fmaf(p.S, f, r.S);
        r.Z = fmaf(f, fmaf(dd, p.S, p.Z), r.Z);
    }
    return r;
}

// The warp's merge of a row's tile partials (lanes over tiles in order, then a fixed
// butterfly), as warp_merge_stats, carrying Z.
__device__ __forceinline__ Stat3 warp_merge_stats3(const float2 *__restrict__ p, const float *__restrict__ z, int n,
                                                   float c, int lane) {
    Stat3 s{-__int_as_float(0x7f800000), 0.f, 0.f};
    for (int q = lane; q < n; q += 32) {
        const float2 ms = __ldcg(p + q);
        s = merge3(s, Stat3{ms.x, ms.y, __ldcg(z + q)}, c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const Stat3 w{__shfl_xor_sync(0xFFFFFFFFu, s.M, o), __shfl_xor_sync(0xFFFFFFFFu, s.S, o),
                      __shfl_xor_sync(0xFFFFFFFFu, s.Z, o)};
        s = merge3(s, w, c);
    }
    return s;
}

// A counter increment that publishes this thread's earlier writes and, for the thread that
// sees the final count, makes the other writers' visible (acquire-release at device scope).
__device__ __forceinline__ int atom_add_acq_rel(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// What the decision of one level needs, gathered by any warp: the merged statistics of the
// level's rows (the target row's Z too for typical acceptance) and the logits at the draft
// token, which the tile pass recorded in xval.  `state` rides along in the first level's
// record.
struct LvStat {
    float2 st, sd;
    float zt, tx, dx;
    int state;
};
template <class D, int RULE>
__device__ __forceinline__ LvStat level_gather(const LevelArgs &a, int64_t seq, int i, int lane) {
    const int G = a.gamma, R = a.R;
    const int64_t rt = seq * R + i, rd = seq * R + G + 1 + i;  // rows of target / draft row i
    const bool has_d = RULE == kRuleSample && i < G;
    LvStat g;
    g.st = make_float2(0.f, 1.f);
    g.sd = make_float2(0.f, 1.f);
    g.zt = g.tx = g.dx = 0.f;
    g.state = 0;
    if (!SV_IN((rt + 1) * a.ntile - 1, int64_t(a.B) * R * a.ntile) ||
        (has_d && !SV_IN((rd + 1) * a.ntile - 1, int64_t(a.B) * R * a.ntile)))
        return g;
    if (i < G) {  // the accept test's operands
        g.tx = __ldcg(a.xval + rt);
        if (has_d) g.dx = __ldcg(a.xval + rd);
    }
    if constexpr (RULE == kRuleTypical) {
        const Stat3 s3 = warp_merge_stats3(a.partial + rt * a.ntile, a.zpart + rt * a.ntile, a.ntile, a.c, lane);
        g.st = make_float2(s3.M, s3.S);
        g.zt = s3.Z;
    } else {
        g.st = warp_merge_stats<true>(a.partial + rt * a.ntile, a.ntile, a.c, lane);
    }
    if (has_d) g.sd = warp_merge_stats<true>(a.partial + rd * a.ntile, a.ntile, a.c, lane);
    return g;
}

// The decision of sequence seq at level i from its gathered record g (one warp); state:
// bit 0 walking, bit 1 marked (0 once the sequence neither walks on nor needs more rows,
// for the rescan).  Returns state != 0.
template <class D, int RULE>
__device__ __forceinline__ bool level_decide(const LevelArgs &a, int64_t seq, int i, int lane, int &state,
                                             const LvStat &g) {
    const int G = a.gamma, R = a.R;
    int *rflag = a.rctl + kRefineCtlWords;
    int32_t *out = a.out_tokens + seq * (G + 1);
    const int64_t rt = seq * R + i, rd = seq * R + G + 1 + i;
    const bool has_d = RULE == kRuleSample && i < G;
    if (!SV_IN(seq, a.B)) {
        state = 0;
        return false;
    }
    const float2 st = g.st, sd = g.sd;
    if (i == 0) {  // the tokens: all in [0, V), else the sequence is invalid
        bool ok = true;
        for (int q = lane; q < G; q += 32) {
            const int32_t xq = a.x[seq * G + q];
            ok &= xq >= 0 && xq < a.V;
        }
        if (!__all_sync(0xFFFFFFFFu, ok)) state = -1;
    }
    if (state >= 0 && (!is_finite(st.x) || (has_d && !is_finite(sd.x)))) {  // not a distribution (R11)
        if (state & 1) {
            state = -1;  // a row the walk reads: the sequence is invalid
        } else {         // a row only the rescan could use: the rows stop here
            state = 0;
            return false;
        }
    }
    if (state < 0) {
        for (int q = lane; q <= G; q += 32) out[q] = -1;
        if (lane == 0) {
            a.accepted_len[seq] = -1;
            a.plan[seq] = make_int2(-1, -1);
            rflag[seq] = 0;
        }
        state = 0;
        return false;
    }
    if (lane == 0) {
        a.rowstat[rt] = st;
        if (has_d) a.rowstat[rd] = sd;
        a.lavail[seq] = i + 1;
        if (i == 0) rflag[seq] = 0;
    }
    if (state & 1) {  // still walking: the accept test of draft i, or the bonus at gamma
        int stop = -1, kind = 0;
        bool near = false;
        if (i < G) {
            const float p = ex2(__fmul_rn(__fsub_rn(g.tx, st.x), a.c)) / st.y;
            bool reject;
            if constexpr (RULE == kRuleSample) {
                const float q = ex2(__fmul_rn(__fsub_rn(g.dx, sd.x), a.c)) / sd.y;
                const float u = uniform01(a.seed, a.offset, uint32_t(seq), uint32_t(i), 0u);
                reject = !(u * q < p);
                near = fabsf(u * q - p) < kRefineAcceptWindow * fmaxf(p, u * q);
            } else if constexpr (RULE == kRuleOnehot) {  // q(x) = 1
                const float u = uniform01(a.seed, a.offset, uint32_t(seq), uint32_t(i), 0u);
                reject = !(u < p);
                near = fabsf(u - p) < kRefineAcceptWindow * fmaxf(p, u);
            } else {  // typical: H = ln S - ln 2 Z / S (natural log, p = 2^a / S)
                const float H = __fsub_rn(logf(st.y), __fdiv_rn(0.69314718f * g.zt, st.y));
                reject = !(p > fminf(a.epsilon, a.delta * expf(-H)));
            }
            if (near) state |= 2;
            if (reject) {
                stop = i;
                kind = RULE == kRuleSample ? 1 : (RULE == kRuleOnehot ? 2 : 0);
            }
        } else {
            stop = G;  // every draft accepted: the bonus from p_gamma
        }
        if (near && lane == 0) rflag[seq] = kRefineAccept;
        if (stop >= 0) {
            for (int q = lane; q <= G; q += 32) {
                if (q < stop) out[q] = a.x[seq * G + q];
                else if (q > stop) out[q] = -1;
            }
            if (lane == 0) {
                a.accepted_len[seq] = stop;
                a.plan[seq] = make_int2(stop, kind);
            }
            state &= ~1;
        }
    }
    return state != 0;
}

constexpr int64_t kSpecBytes = 64 << 20;  // a level fetches every remaining row once that is this little
constexpr float kStepBytes = 32e6f;       // what one more step costs, in bytes streamed (~5 us)
constexpr int kLvWarps = kLvThreads / 32;
constexpr int kLvRecords = 512;  // gathered level records a CTA holds at once

template <class D, bool VEC, int RULE>
__global__ void __launch_bounds__(kLvThreads, 1) level_kernel(LevelArgs a) {
    __shared__ int s_nd;             // sequences this CTA completed in the current chunk
    __shared__ int s_dec[kLvThreads];
    __shared__ LvStat s_lv[kLvRecords];
    griddep_launch_next();
    griddep_wait();  // before any read: the caller's previous kernel may be writing the inputs
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (blockIdx.x == 0 && threadIdx.x < kRefineCtlWords) {  // the draw kernel's re-draw lists and barrier
        a.rctl[threadIdx.x] = 0;
        a.rbar[threadIdx.x] = 0;
    }
    const int G = a.gamma;
    const bool two = RULE == kRuleSample;  // a target and a draft row per level below gamma
    int i = 0, n_prev = a.B, s_prev = 1;
    for (int step = 0; i <= G; ++step) {
        const int n = step == 0 ? a.B : __ldcg(a.lctl + 8 + step);
        if (n == 0) break;  // (the same for every CTA)
        if (!SV_IN(n - 1, a.B)) break;
        const int *list = a.lact + (step & 1) * int64_t(a.B);
        // levels fetched this step: every remaining one once that is little work; else one,
        // and more while the rows read for sequences that will have stopped before them
        // (estimated from the fraction that went on per level so far) stay below what a step
        // of its own costs
        const int left = G + 1 - i;
        const int64_t rows_left = two ? 2 * int64_t(left) - 1 : left;
        int s = 1;
        if (int64_t(n) * rows_left * a.ntile * 4096 <= kSpecBytes) {
            s = left;
        } else if (step > 0) {
            const float go_on = powf(float(n) / float(n_prev), 1.f / float(s_prev));
            const float level_bytes = float(two ? 2 : 1) * float(a.ntile) * 4096.f;
            float waste = 0.f, reach = 1.f;
            while (s < left) {
                reach *= go_on;  // share of the n sequences still walking s levels on
                const float w = float(n) * (1.f - reach) * level_bytes;
                if (waste + w > kStepBytes) break;
                waste += w;
                ++s;
            }
        }
        s = min(s, kLvRecords);  // a sequence's levels of one step fit the CTA's records
        n_prev = n;
        s_prev = s;
        const int nr = two ? 2 * s - (i + s - 1 == G ? 1 : 0) : s;  // rows per sequence this step
        const uint32_t ups = uint32_t(nr) * uint32_t(a.ntile);     // items (tiles) per sequence
        const uint64_t items = uint64_t(n) * ups;
        // item it: the sequence-list entry it / ups, then its rows' tiles in order.  Each CTA
        // takes one contiguous range of items, so it counts its tiles once per sequence it
        // touched instead of once per tile.
        const uint64_t lo = items * blockIdx.x / gridDim.x, hi = items * (blockIdx.x + 1) / gridDim.x;
        auto seq_of = [&](uint32_t ai) { return step == 0 ? int64_t(ai) : int64_t(__ldcg(list + ai)); };
        // The tile loop is software-pipelined: the next item's loads go out before this
        // item's sums.
        uint4 v[kTileVecs];
        int64_t rr = 0, c0 = 0;
        int tile = 0, len = 0, xi = -1;
        auto issue = [&](uint64_t it) {
            const uint32_t ai = uint32_t(it / ups);
            const int local = int(it - uint64_t(ai) * ups);
            const int q = local / a.ntile;
            tile = local - q * a.ntile;
            const int lv = i + (two ? q >> 1 : q);
            const bool is_d = two && (q & 1);
            const int64_t seq = seq_of(ai);
            rr = seq * a.R + (is_d ? G + 1 + lv : lv);
            const char *rp = is_d ? row_ptr(a.d, D::kBytes, seq, lv) : row_ptr(a.t, D::kBytes, seq, lv);
            c0 = int64_t(tile) * tile_elems<D>();
            len = unit_len(a.V, c0, tile_elems<D>());
            xi = lv < G ? __ldg(a.x + seq * G + lv) : -1;  // the draft token whose logit this row gives
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int e0 = (lane + 32 * u) * D::EPV;
                v[u] = e0 < len ? load_vec<D, VEC>(rp, c0, e0, len) : neg_inf_vec<D>();
            }
        };
        if (lo + warp < hi) issue(lo + warp);
        for (uint64_t it = lo + warp; it < hi; it += kLvWarps) {
            const float M = warp_reduce(thread_max<D>(v), [](float x, float y) { return max_nan(x, y); });
            float S = 0.f, Z = 0.f;
            if constexpr (RULE == kRuleTypical) {
                if (is_finite(M)) {
#pragma unroll
                    for (int u = 0; u < kTileVecs; ++u)
#pragma unroll
                        for (int e = 0; e < D::EPV; ++e) {
                            const float y = __fmul_rn(__fsub_rn(vec_elem<D>(v[u], e), M), a.c);
                            const float w = ex2(y);  // 0 for a -inf logit
                            S += w;
                            Z += w > 0.f ? w * y : 0.f;
                        }
                    S = warp_reduce(S, [](float x, float y) { return x + y; });
                    Z = warp_reduce(Z, [](float x, float y) { return x + y; });
                }
            } else {
                if (is_finite(M)) S = warp_reduce(thread_sumexp<D>(v, a.c, M), [](float x, float y) { return x + y; });
            }
            const int64_t slot = rr * a.ntile + tile;
            // the logit at the draft token, if this tile holds it (by the lane that holds it)
            const int64_t xr = int64_t(xi) - c0;
            const int64_t xrow = rr;
            int xl = -1;
            float xv = 0.f;
            if (xi >= 0 && xr >= 0 && xr < len) {
                const int vi = int(xr) / D::EPV, e = int(xr) - vi * D::EPV;  // vector, element in it
                const int wi = D::EPV == 8 ? e >> 1 : e;                         // 32-bit word in the vector
                xl = vi & 31;
                uint32_t w = 0;
#pragma unroll
                for (int u = 0; u < kTileVecs; ++u) {  // (no dynamic index into v: it stays in registers)
                    const uint32_t wu = wi == 0 ? v[u].x : wi == 1 ? v[u].y : wi == 2 ? v[u].z : v[u].w;
                    w = u == (vi >> 5) ? wu : w;
                }
                xv = D::EPV == 8 ? ((e & 1) ? bf16_hi(w) : bf16_lo(w)) : __uint_as_float(w);
            }
            if (it + kLvWarps < hi) issue(it + kLvWarps);
            if (lane == 0 && SV_IN(slot, int64_t(a.B) * a.R * a.ntile)) {
                a.partial[slot] = make_float2(M, S);
                if constexpr (RULE == kRuleTypical) a.zpart[slot] = Z;
            }
            if (lane == xl && SV_IN(xrow, int64_t(a.B) * a.R)) a.xval[xrow] = xv;
        }
        __syncthreads();  // every partial of this CTA's range is written
        // Count this CTA's tiles on the counter of each sequence it touched; the CTA whose count
        // completes a sequence walks its levels of this step (a warp per sequence, in order).
        if (lo < hi) {
            const uint32_t a0 = uint32_t(lo / ups), a1 = uint32_t((hi - 1) / ups);
            for (uint32_t base = a0; base <= a1; base += kLvThreads) {
                if (threadIdx.x == 0) s_nd = 0;
                __syncthreads();
                const uint32_t ai = base + threadIdx.x;
                if (ai <= a1) {
                    const uint64_t b0 = max(lo, uint64_t(ai) * ups), b1 = min(hi, uint64_t(ai + 1) * ups);
                    const int cnt = int(b1 - b0);
                    const int64_t seq = seq_of(ai);
                    int *ctr = a.tcnt + seq;
                    if (SV_IN(seq, a.B) && atom_add_acq_rel(ctr, cnt) + cnt == int(ups)) {
                        *ctr = 0;  // for the next step (after the grid barrier)
                        s_dec[atomicAdd(&s_nd, 1)] = int(seq);
                    }
                }
                __syncthreads();
                // the records of every (sequence, level) this CTA completed, gathered by all
                // warps at once; then a warp per sequence walks its levels in order
                const int nd = s_nd, per_grp = max(1, kLvRecords / s);
                for (int g0 = 0; g0 < nd; g0 += per_grp) {
                    const int ng = min(per_grp, nd - g0);
                    for (int e = warp; e < ng * s; e += kLvWarps) {
                        const int q = e / s, j = e - q * s;
                        const int64_t seq = s_dec[g0 + q];
                        LvStat g = level_gather<D, RULE>(a, seq, i + j, lane);
                        if (j == 0) g.state = i == 0 ? 1 : __ldcg(a.lstate + seq);
                        if (lane == 0) s_lv[e] = g;
                    }
                    __syncthreads();
                    for (int q = warp; q < ng; q += kLvWarps) {
                        const int64_t seq = s_dec[g0 + q];
                        int state = s_lv[q * s].state;
                        bool more = true;
                        for (int j = 0; j < s && more; ++j)
                            more = level_decide<D, RULE>(a, seq, i + j, lane, state, s_lv[q * s + j]);
                        if (lane == 0) {
                            a.lstate[seq] = state;
                            if (more && i + s <= G && SV_IN(step + 1, G + 2)) {
                                const int pos = atomicAdd(a.lctl + 8 + step + 1, 1);
                                if (SV_IN(pos, a.B)) a.lact[((step + 1) & 1) * int64_t(a.B) + pos] = int(seq);
                            }
                        }
                    }
                    __syncthreads();
                }
                __syncthreads();  // s_nd is reset for the next chunk
            }
        }
        if (!grid_barrier(a.lctl)) {
            if (threadIdx.x == 0) atomicExch(a.rctl + kRefineStatus, int(SV_ERR_TIMEOUT));
            return;
        }
        i += s;
    }
}

}  // namespace

cudaError_t launch_level(int rule, int dtype, bool vec, const LevelArgs &a, cudaStream_t s) {
    void (*k)(LevelArgs) = nullptr;
    if (rule == kRuleSample) k = dtype == 1 ? (vec ? level_kernel<BF16, true, kRuleSample> : level_kernel<BF16, false, kRuleSample>)
                                            : (vec ? level_kernel<F32, true, kRuleSample> : level_kernel<F32, false, kRuleSample>);
    else if (rule == kRuleOnehot) k = dtype == 1 ? (vec ? level_kernel<BF16, true, kRuleOnehot> : level_kernel<BF16, false, kRuleOnehot>)
                                                 : (vec ? level_kernel<F32, true, kRuleOnehot> : level_kernel<F32, false, kRuleOnehot>);
    else k = dtype == 1 ? (vec ? level_kernel<BF16, true, kRuleTypical> : level_kernel<BF16, false, kRuleTypical>)
                        : (vec ? level_kernel<F32, true, kRuleTypical> : level_kernel<F32, false, kRuleTypical>);
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kLvThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    e = cudaMemsetAsync(a.lctl, 0, sizeof(int) * size_t(8 + a.gamma + 2), s);  // barrier words, level counts
    if (e == cudaSuccess) e = cudaMemsetAsync(a.tcnt, 0, sizeof(int) * size_t(a.B), s);
    if (e != cudaSuccess) return e;
    return launch_after_ex(true, k, unsigned(sms), kLvThreads, 0, s, a);
}

}  // namespace sv
