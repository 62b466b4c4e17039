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
//   stats_partial   every (row, 32 KB chunk) of the 2 gamma + 1 rows of every sequence:
//                   NaN-propagating max M and sum 2^((l - M) log2(e) / T), one CTA each.
//   decide          one warp per sequence: merge the chunk partials into (M, S) per row,
//                   gather p_i(x_i), q_i(x_i), draw the Philox uniforms and scan.
//   residual_chunks (sequences that rejected) the residual mass of every chunk of row k.
//   locate          one CTA per sequence: prefix over chunk masses, then an in-order block
//                   scan inside the chosen chunk; first j with C_j > u' R.
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

__device__ __forceinline__ const char *row_ptr(const Logits &L, int bytes, int64_t b, int64_t r) {
    return static_cast<const char *>(L.ptr) + (b * L.batch_stride + r * L.row_stride) * bytes;
}

template <class D>
__device__ __forceinline__ uint4 neg_inf_vec() {
    return make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
}

// Unnormalised target weight 2^((t - M) c) = exp((t - M) / T) with a single rounding of
// the (exact) difference times c.
__device__ __forceinline__ float weight(float x, float M, float c) {
    return ex2(__fmul_rn(__fsub_rn(x, M), c));
}

// (p_j - q_j)+ with p_j = 2^((t_j - M_t) c) / S_t and q_j likewise.  Both the chunk-mass
// kernel and the in-chunk scan call this one function, so the two agree bit for bit.  The
// products and the difference are explicitly rounded (no FMA contraction), so rows that
// are identical give exactly p_j - q_j = 0, as in exact arithmetic.
__device__ __forceinline__ float residual_weight(float tj, float dj, float c, float mt, float inv_st,
                                                 float md, float inv_sd) {
    const float p = __fmul_rn(weight(tj, mt, c), inv_st);
    const float q = __fmul_rn(weight(dj, md, c), inv_sd);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// ------------------------------------------------------------------------------------
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 4)
    stats_partial_kernel(Logits a, int rows_a, Logits bt, int R, int V, int nchunk, float c,
                         float2 *__restrict__ partial) {
    __shared__ float2 red[kWarps];
    const int64_t item = blockIdx.x;
    const int64_t row = item / nchunk;
    const int chunk = int(item - row * nchunk);
    const int64_t seq = row / R;
    const int local = int(row - seq * R);
    const char *rp = local < rows_a ? row_ptr(a, D::kBytes, seq, local)
                                    : row_ptr(bt, D::kBytes, seq, local - rows_a);
    const int64_t c0 = int64_t(chunk) * chunk_elems<D>();
    const int len = chunk_len<D>(V, c0);

    uint4 v[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        const int e0 = (threadIdx.x + u * kThreads) * D::EPV;
        v[u] = e0 < len ? load_vec<D, VEC>(rp, c0, e0, len) : neg_inf_vec<D>();
    }
    const float m = thread_max<D>(v);
    const float S = is_finite(m) ? thread_sumexp<D>(v, c, m) : 0.f;
    const float2 r = block_reduce(
        make_float2(m, S), [c](float2 x, float2 y) { return merge_stats(x, y, c); }, red);
    if (threadIdx.x == 0) partial[item] = r;
}

// ------------------------------------------------------------------------------------
template <class D>
__global__ void __launch_bounds__(128)
    decide_kernel(Logits t, Logits d, int B, int gamma, int V, int nchunk, float c,
                  const int32_t *__restrict__ x, uint64_t seed, uint64_t offset,
                  const float2 *__restrict__ partial, float2 *__restrict__ rowstat,
                  int2 *__restrict__ plan, int32_t *__restrict__ accepted_len,
                  int32_t *__restrict__ out_tokens) {
    const int lane = threadIdx.x & 31;
    const int64_t seq = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (seq >= B) return;
    const int R = 2 * gamma + 1;

    bool ok = true;
    for (int r = lane; r < R; r += 32) {
        const float2 *p = partial + (seq * R + r) * nchunk;
        float2 s = p[0];
        for (int ch = 1; ch < nchunk; ++ch) s = merge_stats(s, p[ch], c);
        rowstat[seq * R + r] = s;
        ok &= is_finite(s.x);
    }
    for (int i = lane; i < gamma; i += 32) {
        const int32_t xi = x[seq * gamma + i];
        ok &= xi >= 0 && xi < V;
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    int32_t *out = out_tokens + seq * (gamma + 1);
    if (!ok) {
        for (int i = lane; i <= gamma; i += 32) out[i] = -1;
        if (lane == 0) {
            accepted_len[seq] = -1;
            plan[seq] = make_int2(-1, -1);
        }
        return;
    }
    __syncwarp();  // rowstat written by other lanes of this warp is read below

    int k = gamma;
    for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        bool reject = false;
        if (i < gamma) {
            const int32_t xi = x[seq * gamma + i];
            const float2 st = rowstat[seq * R + i];
            const float2 sd = rowstat[seq * R + gamma + 1 + i];
            const float tx = load_elem<D>(row_ptr(t, D::kBytes, seq, i), xi);
            const float dx = load_elem<D>(row_ptr(d, D::kBytes, seq, i), xi);
            const float p = weight(tx, st.x, c) / st.y;
            const float q = weight(dx, sd.x, c) / sd.y;
            const float u = uniform01(seed, offset, uint32_t(seq), uint32_t(i), 0u);
            reject = !(u * q < p);
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, reject);
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
    }
}

// ------------------------------------------------------------------------------------
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 2)
    residual_chunks_kernel(Logits t, Logits d, int gamma, int V, int nchunk, float c,
                           const float2 *__restrict__ rowstat, const int2 *__restrict__ plan,
                           float *__restrict__ csum) {
    __shared__ float red[kWarps];
    const int64_t item = blockIdx.x;
    const int64_t seq = item / nchunk;
    const int chunk = int(item - seq * nchunk);
    const int2 pl = plan[seq];
    if (pl.y != 1) return;  // uniform over the block
    const int k = pl.x, R = 2 * gamma + 1;
    const float2 st = rowstat[seq * R + k], sd = rowstat[seq * R + gamma + 1 + k];
    const float inv_st = 1.f / st.y, inv_sd = 1.f / sd.y;
    const char *tp = row_ptr(t, D::kBytes, seq, k);
    const char *dp = row_ptr(d, D::kBytes, seq, k);
    const int64_t c0 = int64_t(chunk) * chunk_elems<D>();
    const int len = chunk_len<D>(V, c0);

    uint4 tv[kVecPerThread], dv[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        const int e0 = (threadIdx.x + u * kThreads) * D::EPV;
        tv[u] = e0 < len ? load_vec<D, VEC>(tp, c0, e0, len) : neg_inf_vec<D>();
        dv[u] = e0 < len ? load_vec<D, VEC>(dp, c0, e0, len) : neg_inf_vec<D>();
    }
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u)
#pragma unroll
        for (int e = 0; e < D::EPV; ++e)
            acc += residual_weight(vec_elem<D>(tv[u], e), vec_elem<D>(dv[u], e), c, st.x, inv_st,
                                   sd.x, inv_sd);
    const float s = block_reduce(acc, [](float a, float b) { return a + b; }, red);
    if (threadIdx.x == 0) csum[item] = s;
}

// ------------------------------------------------------------------------------------
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads)
    locate_kernel(Logits t, Logits d, int gamma, int V, int nchunk, float c, uint64_t seed,
                  uint64_t offset, const float2 *__restrict__ partial,
                  const float2 *__restrict__ rowstat, const int2 *__restrict__ plan,
                  const float *__restrict__ csum, int32_t *__restrict__ out_tokens) {
    __shared__ float fsc[kWarps];
    __shared__ int isc[kWarps];
    __shared__ float hit_base;
    const int64_t seq = blockIdx.x;
    const int2 pl = plan[seq];
    if (pl.y < 0) return;  // invalid sequence: outputs already written by decide
    const int k = pl.x, R = 2 * gamma + 1;
    int mode = pl.y;  // 1: residual after a rejection, 0: bonus draw from p
    const float2 st = rowstat[seq * R + k];
    const float2 sd = mode ? rowstat[seq * R + gamma + 1 + k] : make_float2(0.f, 1.f);
    const float inv_st = 1.f / st.y, inv_sd = 1.f / sd.y;
    const float2 *prow = partial + (seq * R + k) * nchunk;
    const float *crow = csum + seq * nchunk;
    auto chunk_mass = [&](int ch) -> float {
        if (ch >= nchunk) return 0.f;
        if (mode) return crow[ch];
        const float2 p = prow[ch];
        return p.y * weight(p.x, st.x, c);  // mass of chunk ch under 2^((l - M) c)
    };

    // total mass R (as the deterministic tile-by-tile scan computes it)
    float total = 0.f;
    for (int pass = 0; pass < 2; ++pass) {
        total = 0.f;
        for (int base = 0; base < nchunk; base += kThreads) {
            float tt;
            block_inclusive_scan(chunk_mass(base + threadIdx.x), fsc, &tt);
            total += tt;
        }
        if (mode == 1 && !(total > 0.f)) mode = 0;  // exact-zero residual: draw from p
        else break;
    }
    const float thr = uniform01(seed, offset, uint32_t(seq), uint32_t(k), 1u) * total;

    // the chunk holding the threshold: first ch with C_ch > thr (C inclusive)
    int cstar = -1;
    bool force_last = false;
    float carry = 0.f;
    int last_pos_chunk = -1;
    float last_pos_base = 0.f;
    for (int base = 0; base < nchunk && cstar < 0; base += kThreads) {
        const int ch = base + threadIdx.x;
        const float w = chunk_mass(ch);
        float tt;
        const float incl = block_inclusive_scan(w, fsc, &tt);
        const bool hit = ch < nchunk && carry + incl > thr;
        const int first = block_reduce(hit ? ch : kNoIndex, [](int a, int b) { return min(a, b); }, isc);
        const int lp = block_reduce((ch < nchunk && w > 0.f) ? ch : -1,
                                    [](int a, int b) { return max(a, b); }, isc);
        if (first != kNoIndex) {
            if (ch == first) hit_base = carry + incl - w;
            __syncthreads();
            cstar = first;
            carry = hit_base;
        } else {
            if (lp >= 0) {
                if (ch == lp) hit_base = carry + incl - w;
                __syncthreads();
                last_pos_chunk = lp;
                last_pos_base = hit_base;
            }
            carry += tt;
        }
        __syncthreads();
    }
    if (cstar < 0) {  // rounding left the threshold above the last prefix
        cstar = last_pos_chunk >= 0 ? last_pos_chunk : 0;
        carry = last_pos_base;
        force_last = true;
    }

    // in-order scan inside chunk cstar: thread t owns elements [t*EPT, (t+1)*EPT)
    constexpr int EPT = kVecPerThread * D::EPV;
    const char *tp = row_ptr(t, D::kBytes, seq, k);
    const char *dp = mode ? row_ptr(d, D::kBytes, seq, k) : nullptr;
    const int64_t c0 = int64_t(cstar) * chunk_elems<D>();
    const int len = chunk_len<D>(V, c0);
    float r[EPT];
    float tsum = 0.f;
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
        const int e0 = (threadIdx.x * kVecPerThread + u) * D::EPV;
        const uint4 tv = e0 < len ? load_vec<D, VEC>(tp, c0, e0, len) : neg_inf_vec<D>();
        uint4 dv = neg_inf_vec<D>();
        if (mode && e0 < len) dv = load_vec<D, VEC>(dp, c0, e0, len);
#pragma unroll
        for (int e = 0; e < D::EPV; ++e) {
            const float tj = vec_elem<D>(tv, e);
            const float w = mode ? residual_weight(tj, vec_elem<D>(dv, e), c, st.x, inv_st, sd.x, inv_sd)
                                 : weight(tj, st.x, c);
            r[u * D::EPV + e] = w;
            tsum += w;
        }
    }
    float tt;
    const float incl = block_inclusive_scan(tsum, fsc, &tt);
    float P = carry + (incl - tsum);
    int cand = kNoIndex, lastpos = -1;
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
        const int j = threadIdx.x * EPT + q;
        P += r[q];
        if (j < len) {
            if (!force_last && cand == kNoIndex && P > thr) cand = j;
            if (r[q] > 0.f) lastpos = j;
        }
    }
    cand = block_reduce(cand, [](int a, int b) { return min(a, b); }, isc);
    lastpos = block_reduce(lastpos, [](int a, int b) { return max(a, b); }, isc);
    int tok = cand != kNoIndex ? cand : lastpos;
    if (tok < 0) tok = 0;
    if (threadIdx.x == 0) out_tokens[seq * (gamma + 1) + k] = int32_t(c0 + tok);
}

// ------------------------------------------------------------------------------------
__global__ void rowstats_finalize_kernel(int rows, int nchunk, float c, float inv_t,
                                         const float2 *__restrict__ partial, float *__restrict__ m_out,
                                         float *__restrict__ lse_out) {
    const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const float2 *p = partial + r * nchunk;
    float2 s = p[0];
    for (int ch = 1; ch < nchunk; ++ch) s = merge_stats(s, p[ch], c);
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
#define SV_DISPATCH(DTYPE, VEC, KERNEL, GRID, BLOCK, STREAM, ...)                                  \
    do {                                                                                         \
        if ((DTYPE) == 1) {                                                                      \
            if (VEC) KERNEL<BF16, true><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);                \
            else KERNEL<BF16, false><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);                   \
        } else {                                                                                 \
            if (VEC) KERNEL<F32, true><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);                 \
            else KERNEL<F32, false><<<GRID, BLOCK, 0, STREAM>>>(__VA_ARGS__);                    \
        }                                                                                        \
    } while (0)

cudaError_t launch_stats_partial(int dtype, bool vec, Logits a, int rows_a, Logits b, int R, int B,
                                 int V, int nchunk, float c, void *partial, cudaStream_t s) {
    const unsigned grid = unsigned(int64_t(B) * R * nchunk);
    SV_DISPATCH(dtype, vec, stats_partial_kernel, grid, kThreads, s, a, rows_a, b, R, V, nchunk, c,
                static_cast<float2 *>(partial));
    return cudaGetLastError();
}

cudaError_t launch_decide(int dtype, Logits t, Logits d, int B, int gamma, int V, int nchunk,
                          float c, const int32_t *x, uint64_t seed, uint64_t offset,
                          const void *partial, void *rowstat, void *plan, int32_t *accepted_len,
                          int32_t *out_tokens, cudaStream_t s) {
    const unsigned grid = unsigned((int64_t(B) * 32 + 127) / 128);
    if (dtype == 1)
        decide_kernel<BF16><<<grid, 128, 0, s>>>(t, d, B, gamma, V, nchunk, c, x, seed, offset,
                                                 static_cast<const float2 *>(partial),
                                                 static_cast<float2 *>(rowstat), static_cast<int2 *>(plan),
                                                 accepted_len, out_tokens);
    else
        decide_kernel<F32><<<grid, 128, 0, s>>>(t, d, B, gamma, V, nchunk, c, x, seed, offset,
                                                static_cast<const float2 *>(partial),
                                                static_cast<float2 *>(rowstat), static_cast<int2 *>(plan),
                                                accepted_len, out_tokens);
    return cudaGetLastError();
}

cudaError_t launch_residual_chunks(int dtype, bool vec, Logits t, Logits d, int B, int gamma,
                                   int V, int nchunk, float c, const void *rowstat,
                                   const void *plan, float *csum, cudaStream_t s) {
    const unsigned grid = unsigned(int64_t(B) * nchunk);
    SV_DISPATCH(dtype, vec, residual_chunks_kernel, grid, kThreads, s, t, d, gamma, V, nchunk, c,
                static_cast<const float2 *>(rowstat), static_cast<const int2 *>(plan), csum);
    return cudaGetLastError();
}

cudaError_t launch_locate(int dtype, bool vec, Logits t, Logits d, int B, int gamma, int V,
                          int nchunk, float c, uint64_t seed, uint64_t offset, const void *partial,
                          const void *rowstat, const void *plan, const float *csum,
                          int32_t *out_tokens, cudaStream_t s) {
    SV_DISPATCH(dtype, vec, locate_kernel, unsigned(B), kThreads, s, t, d, gamma, V, nchunk, c, seed,
                offset, static_cast<const float2 *>(partial), static_cast<const float2 *>(rowstat),
                static_cast<const int2 *>(plan), csum, out_tokens);
    return cudaGetLastError();
}

cudaError_t launch_rowstats_finalize(int rows, int nchunk, float c, float inv_t, const void *partial,
                                     float *m_out, float *lse_out, cudaStream_t s) {
    const unsigned grid = unsigned((int64_t(rows) + 255) / 256);
    rowstats_finalize_kernel<<<grid, 256, 0, s>>>(rows, nchunk, c, inv_t,
                                                  static_cast<const float2 *>(partial), m_out, lse_out);
    return cudaGetLastError();
}

cudaError_t launch_uniforms(uint64_t seed, uint64_t offset, int B, int positions, int purpose,
                            float *out, cudaStream_t s) {
    const int64_t n = int64_t(B) * positions;
    const unsigned grid = unsigned((n + 255) / 256);
    uniforms_kernel<<<grid, 256, 0, s>>>(seed, offset, B, positions, purpose, out);
    return cudaGetLastError();
}

}  // namespace sv
