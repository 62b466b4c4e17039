// sv_greedy.cu -- greedy and greedy token-tree verification.
//
// Method: temperature 0 turns p and q into point masses, so the accept rule becomes
// "accept while the draft equals the target argmax" and the token at the first mismatch
// (or after the last draft) is that row's argmax ("7.6 Speculative Decoding: Draft Models,
// Medusa, EAGLE & Lookahead": "Extending to a chain of gamma draft tokens"; "Medusa, EAGLE
// and self-speculation": speculative_greedy).  For a token tree, a node is kept when its
// token is the argmax of its parent's row and its parent is kept; the deepest kept node
// ends the path and its own row's argmax is the bonus (same page, "Tree Attention" and
// Exercise 5, verify_tree_greedy).
//
// GPU decomposition:
//   max_tiles        persistent: every 4 KB tile of every row, one warp per tile: the
//                    tile's NaN-propagating maximum.
//   greedy_finalize  one CTA per sequence, one warp per row: the row maximum and the lowest
//                    tile holding it, then the first position of that value inside that one
//                    tile (re-read, 4 KB); then the longest matching prefix.
//   tree_finalize    one CTA per sequence: the same argmax for all N nodes, validate the
//                    tree, accepted flags by walking each node's root path, deepest node
//                    (lowest index on ties), write the path.
// Searching for the index only inside the winning tile keeps the streaming pass as cheap
// as a plain maximum.
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads, 4)
    max_tiles_kernel(Logits t, int R, int V, int ntile, int64_t items, float *__restrict__ partial) {
    griddep_launch_next();
    griddep_wait();  // before any read: the caller's previous kernel may be writing the logits
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = int64_t(gridDim.x) * kWarps;
    for (TileWalk w(int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5), nwarps, R, ntile); w.it < items;
         w.next(nwarps)) {
        const char *rp = row_ptr(t, D::kBytes, w.seq, w.local);
        const int64_t c0 = int64_t(w.tile) * tile_elems<D>();
        const int len = unit_len(V, c0, tile_elems<D>());
        uint4 v[kTileVecs];
#pragma unroll
        for (int u = 0; u < kTileVecs; ++u) {
            const int e0 = (lane + 32 * u) * D::EPV;
            v[u] = e0 < len ? load_vec<D, VEC>(rp, c0, e0, len)
                            : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
        }
        const float m = warp_reduce(thread_max<D>(v), [](float a, float b) { return max_nan(a, b); });
        if (lane == 0 && SV_IN(w.it, items)) partial[w.it] = m;
    }
}

// The argmax of one row (one warp; every lane returns it): the largest tile maximum, on
// ties the lowest tile (a NaN maximum marks bad data and absorbs everything), then the
// first position of that value inside that tile, read again from the row.  Returns (value
// bits, index).
template <class D, bool VEC>
__device__ int2 warp_row_argmax(const float *__restrict__ tmax, int ntile, const char *row, int V, int lane) {
    int2 best = make_int2(__float_as_int(-__int_as_float(0x7f800000)), kNoIndex);
    for (int q0 = lane; q0 < ntile; q0 += 128) {
        float e[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) e[j] = q0 + 32 * j < ntile ? tmax[q0 + 32 * j] : -__int_as_float(0x7f800000);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (q0 + 32 * j < ntile) best = merge_argmax(best, make_int2(__float_as_int(e[j]), q0 + 32 * j));
    }
    best = warp_reduce(best, [](int2 a, int2 b) { return merge_argmax(a, b); });
    const float bm = __int_as_float(best.x);
    if (bm != bm) return make_int2(best.x, -1);
    const int64_t c0 = int64_t(best.y) * tile_elems<D>();
    const int len = unit_len(V, c0, tile_elems<D>());
    uint4 v[kTileVecs];
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int e0 = (lane + 32 * u) * D::EPV;
        v[u] = e0 < len ? load_vec<D, VEC>(row, c0, e0, len)
                        : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
    }
    // lane-local first match (lane l holds vectors l, l + 32, ... in index order), then the
    // lowest over the lanes; reverse scans with selects keep the lowest match
    int idx = kNoIndex;
#pragma unroll
    for (int u = kTileVecs - 1; u >= 0; --u) {
        const int e0 = (lane + 32 * u) * D::EPV;
#pragma unroll
        for (int e = D::EPV - 1; e >= 0; --e) {
            const bool hit = vec_elem<D>(v[u], e) == bm && e0 + e < len;
            idx = hit ? int(c0) + e0 + e : idx;
        }
    }
    idx = warp_reduce(idx, [](int a, int b) { return min(a, b); });
    return make_int2(best.x, idx);
}

// Greedy finalize, one CTA per sequence: warp w finds the argmax of rows w, w + 8, ...;
// warp 0 then finds the longest matching prefix.
template <class D, bool VEC>
__global__ void __launch_bounds__(kThreads)
    greedy_finalize_kernel(Logits t, int B, int gamma, int V, int ntile, const float *__restrict__ partial,
                           const int32_t *__restrict__ x, int32_t *__restrict__ accepted_len,
                           int32_t *__restrict__ out_tokens) {
    extern __shared__ int2 s_best[];  // [gamma + 1]
    griddep_launch_next();
    griddep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t seq = blockIdx.x;
    const int R = gamma + 1;
    for (int i = warp; i < R; i += kWarps) {
        if (!SV_IN((seq * R + i + 1) * ntile - 1, int64_t(B) * R * ntile)) continue;
        const int2 best = warp_row_argmax<D, VEC>(partial + (seq * R + i) * ntile, ntile,
                                                  row_ptr(t, D::kBytes, seq, i), V, lane);
        if (lane == 0) s_best[i] = best;
    }
    __syncthreads();
    if (warp != 0) return;
    bool ok = true;
    for (int i = lane; i < R; i += 32) {
        const float v = __int_as_float(s_best[i].x);
        ok &= v == v;
    }
    for (int i = lane; i < gamma; i += 32) {
        const int32_t xi = x[seq * gamma + i];
        ok &= xi >= 0 && xi < V;
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    int32_t *out = out_tokens + seq * R;
    if (!ok) {
        for (int i = lane; i < R; i += 32) out[i] = -1;
        if (lane == 0) accepted_len[seq] = -1;
        return;
    }
    int n = gamma;
    for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        const bool miss = i < gamma && x[seq * gamma + i] != s_best[i].y;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, miss);
        if (m) {
            n = i0 + __ffs(m) - 1;
            break;
        }
    }
    if (!SV_IN(n, R)) return;
    for (int i = lane; i < R; i += 32) out[i] = i < n ? x[seq * gamma + i] : (i == n ? s_best[n].y : -1);
    if (lane == 0) accepted_len[seq] = n;
}

constexpr int kTreeThreads = 512;
constexpr int kKeyShift = 11;  // node index < 2^11 (SV_MAX_TREE_NODES = 1024)

template <class D, bool VEC>
__global__ void __launch_bounds__(kTreeThreads)
    tree_finalize_kernel(Logits t, int B, int N, int V, int ntile, const float *__restrict__ partial,
                         const int32_t *__restrict__ parent, const int32_t *__restrict__ node_tokens,
                         int max_depth, int32_t *__restrict__ accepted_len,
                         int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_path) {
    extern __shared__ int s_tree[];  // a[N], par[N], tok[N]
    constexpr int kTreeWarps = kTreeThreads / 32;
    __shared__ int red[kTreeWarps];
    griddep_launch_next();
    int *a = s_tree, *par = s_tree + N, *tok = s_tree + 2 * N;
    const int64_t seq = blockIdx.x;
    const int W = max_depth + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int tree_ok = 1, seq_ok = 1;
    for (int v = threadIdx.x; v < N; v += kTreeThreads) {  // inputs of the call: before the wait
        const int p = parent[v];
        par[v] = p;
        tree_ok &= v == 0 ? p == -1 : (p >= 0 && p < v);
        const int tk = node_tokens[seq * N + v];
        tok[v] = tk;
        if (v > 0) seq_ok &= tk >= 0 && tk < V;
    }
    griddep_wait();
    for (int v = warp; v < N; v += kTreeWarps) {  // node v's argmax: one warp per row
        if (!SV_IN((seq * N + v + 1) * ntile - 1, int64_t(B) * N * ntile)) continue;
        const int2 best = warp_row_argmax<D, VEC>(partial + (seq * N + v) * ntile, ntile,
                                                  row_ptr(t, D::kBytes, seq, v), V, lane);
        if (lane == 0) {
            const float val = __int_as_float(best.x);
            seq_ok &= val == val;
            a[v] = best.y;
        }
    }
    tree_ok = __syncthreads_and(tree_ok);
    seq_ok = __syncthreads_and(seq_ok);

    int best_key = -1, max_d = 0;
    if (tree_ok) {  // parents precede children, so every walk ends at the root
        for (int v = threadIdx.x; v < N; v += kTreeThreads) {
            int d = 0, w = v;
            bool kept = true;
            while (w != 0) {
                const int p = par[w];
                if (!SV_IN(p, N)) break;
                kept = kept && tok[w] == a[p];
                w = p;
                ++d;
            }
            max_d = max(max_d, d);
            if (kept) best_key = max(best_key, (d << kKeyShift) | ((1 << kKeyShift) - 1 - v));
        }
    }
    max_d = block_reduce<kTreeWarps>(max_d, [](int x, int y) { return max(x, y); }, red);
    best_key = block_reduce<kTreeWarps>(best_key, [](int x, int y) { return max(x, y); }, red);
    if (threadIdx.x != 0) return;

    int32_t *out = out_tokens + seq * W;
    int32_t *path = out_path ? out_path + seq * W : nullptr;
    if (!tree_ok || !seq_ok || max_d > max_depth) {
        for (int s = 0; s < W; ++s) {
            out[s] = -1;
            if (path) path[s] = -1;
        }
        accepted_len[seq] = -1;
        return;
    }
    const int d = best_key >> kKeyShift;
    const int vstar = (1 << kKeyShift) - 1 - (best_key & ((1 << kKeyShift) - 1));
    if (!SV_IN(vstar, N) || !SV_IN(d, W)) return;
    for (int s = d + 1; s < W; ++s) {
        out[s] = -1;
        if (path) path[s] = -1;
    }
    out[d] = a[vstar];  // the bonus: argmax of the deepest kept node's row
    for (int s = d, w = vstar; s >= 0; --s) {
        if (!SV_IN(w, N)) break;
        if (path) path[s] = w;
        if (s >= 1) out[s - 1] = tok[w];
        w = par[w];
    }
    accepted_len[seq] = d;
}

}  // namespace

cudaError_t launch_max_tiles(int dtype, bool vec, Logits t, int R, int B, int V, int ntile, void *partial,
                             cudaStream_t s) {
    const int64_t items = int64_t(B) * R * ntile;
    auto k = dtype == 1 ? (vec ? max_tiles_kernel<BF16, true> : max_tiles_kernel<BF16, false>)
                        : (vec ? max_tiles_kernel<F32, true> : max_tiles_kernel<F32, false>);
    unsigned grid = 0;
    cudaError_t e = persistent_grid(k, items, &grid);
    if (e != cudaSuccess) return e;
    return launch_after(k, grid, kThreads, 0, s, t, R, V, ntile, items, static_cast<float *>(partial));
}

cudaError_t launch_greedy_finalize(int dtype, bool vec, Logits t, int B, int gamma, int V, int ntile,
                                   const void *partial, const int32_t *x, int32_t *accepted_len,
                                   int32_t *out_tokens, cudaStream_t s) {
    const size_t smem = size_t(gamma + 1) * sizeof(int2);
    auto k = dtype == 1 ? (vec ? greedy_finalize_kernel<BF16, true> : greedy_finalize_kernel<BF16, false>)
                        : (vec ? greedy_finalize_kernel<F32, true> : greedy_finalize_kernel<F32, false>);
    return launch_after(k, unsigned(B), kThreads, smem, s, t, B, gamma, V, ntile,
                        static_cast<const float *>(partial), x, accepted_len, out_tokens);
}

cudaError_t launch_tree_finalize(int dtype, bool vec, Logits t, int B, int N, int V, int ntile,
                                 const void *partial, const int32_t *parent, const int32_t *node_tokens,
                                 int max_depth, int32_t *accepted_len, int32_t *out_tokens, int32_t *out_path,
                                 cudaStream_t s) {
    const size_t smem = size_t(3) * N * sizeof(int);
    auto k = dtype == 1 ? (vec ? tree_finalize_kernel<BF16, true> : tree_finalize_kernel<BF16, false>)
                        : (vec ? tree_finalize_kernel<F32, true> : tree_finalize_kernel<F32, false>);
    return launch_after(k, unsigned(B), kTreeThreads, smem, s, t, B, N, V, ntile,
                        static_cast<const float *>(partial), parent, node_tokens, max_depth, accepted_len,
                        out_tokens, out_path);
}

}  // namespace sv
