// sv_lazy.cu -- lazy greedy verification: read only the rows whose argmax decides something.
//
// Method ("7.6 Speculative Decoding: Draft Models, Medusa, EAGLE & Lookahead", "Extending
// to a chain" at temperature 0 and "Tree Attention" / Exercise 5 verify_tree_greedy; the
// greedy rule of "Medusa, EAGLE and self-speculation", speculative_greedy): node v != 0 is
// accepted when its token equals the argmax of its parent's row and its parent is
// accepted; the deepest accepted node (lowest index among equally deep ones) ends the path
// and its row's argmax is the bonus.  A chain is the tree whose node v has parent v - 1.
//
// Only accepted nodes' rows can change the result (a row decides its children's
// acceptance and, for the deepest accepted node, the bonus), so a cluster of CS CTAs per
// sequence (CS = 1 .. 8, as many SMs as the batch leaves for each sequence) walks the
// accepted nodes in index order -- parents come before children -- and reads exactly those
// rows, each CTA its share of a row's tiles.  Each row's argmax is the two-step search of
// the full path: the largest 4 KB-tile maximum (lowest tile on ties, NaN absorbing), merged
// over the cluster through distributed shared memory, then the first position of that value
// inside that tile, found by the warp that read it.
#include "sv_checks.cuh"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kLzThreads = 1024;
constexpr int kLzWarps = kLzThreads / 32;

}  // namespace

// chain: parent(v) = v - 1 and node v's token is tokens[seq * (N - 1) + v - 1] (draft
// tokens [B][gamma], N = gamma + 1); otherwise parent[N] and node_tokens [B][N].
template <class D, bool VEC, int CS>
__global__ void __launch_bounds__(kLzThreads, 1)
    greedy_walk_kernel(Logits t, int N, int V, bool chain, const int32_t *__restrict__ parent,
                       const int32_t *__restrict__ tokens, int max_depth, int32_t *__restrict__ accepted_len,
                       int32_t *__restrict__ out_tokens, int32_t *__restrict__ out_path) {
    extern __shared__ int s_int[];
    int *s_par = s_int, *s_tok = s_int + N, *s_dep = s_int + 2 * N, *s_acc = s_int + 3 * N;
    int *s_arg = s_int + 4 * N;  // argmax of each accepted node's row
    int *s_path = s_int + 5 * N;  // max_depth + 1
    __shared__ int2 s_best[kLzWarps];
    __shared__ int s_cbest[2];  // this CTA's best (max bits, tile) of the current row
    __shared__ int s_flag, s_idx;
    griddep_launch_next();
    griddep_wait();  // the caller's kernels may still be writing the inputs
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = cluster_rank<CS>();
    const int64_t seq = blockIdx.x / CS;
    const int W = max_depth + 1;
    int32_t *out = out_tokens + seq * W;
    int32_t *opath = out_path ? out_path + seq * W : nullptr;
    constexpr int TE = tile_elems<D>();
    const int ntile = int((int64_t(V) + TE - 1) / TE);
    const bool writer = rank == 0;  // one CTA of the cluster writes the outputs

    if (tid == 0) s_flag = 1;
    __syncthreads();
    for (int v = tid; v < N; v += kLzThreads) {
        const int p = chain ? v - 1 : parent[v];
        const int tk = v == 0 ? 0 : (chain ? tokens[seq * (N - 1) + v - 1] : tokens[seq * N + v]);
        s_par[v] = p;
        s_tok[v] = tk;
        s_acc[v] = v == 0;
        if ((v == 0 && p != -1) || (v > 0 && (p < 0 || p >= v)) || tk < 0 || tk >= V) s_flag = 0;
    }
    __syncthreads();
    if (s_flag) {
        for (int v = tid; v < N; v += kLzThreads) {
            int dpt = 0;
            for (int w = v; w != 0 && dpt <= max_depth && SV_IN(w, N); w = s_par[w]) ++dpt;
            s_dep[v] = dpt;
            if (dpt > max_depth) s_flag = 0;
        }
    }
    __syncthreads();
    auto fail = [&]() {
        if (!writer) return;
        for (int i = tid; i < W; i += kLzThreads) {
            out[i] = -1;
            if (opath) opath[i] = -1;
        }
        if (tid == 0) accepted_len[seq] = -1;
    };
    if (!s_flag) {  // (the same in every CTA of the cluster: no shared memory was read remotely)
        fail();
        return;
    }

    // The argmax of row v (every thread returns it; -1 for a row with a NaN).  Warp g of the
    // cluster (g = rank * kLzWarps + warp) takes tiles g, g + CS * kLzWarps, ...; it keeps
    // its last tile, which is its only one whenever the row has at most CS * kLzWarps tiles.
    const int gwarp = rank * kLzWarps + warp;
    auto row_argmax = [&](int v) -> int {
        const char *row = row_ptr(t, D::kBytes, seq, v);
        int2 best = make_int2(__float_as_int(-__int_as_float(0x7f800000)), kNoIndex);  // (max bits, tile)
        uint4 vv[kTileVecs];
        int held = -1;  // the tile whose logits vv holds
        for (int tile = gwarp; tile < ntile; tile += CS * kLzWarps) {
            const int64_t c0 = int64_t(tile) * TE;
            const int len = unit_len(V, c0, TE);
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int e0 = (lane + 32 * u) * D::EPV;
                vv[u] = e0 < len ? load_vec<D, VEC>(row, c0, e0, len) : neg_inf_vec<D>();
            }
            held = tile;
            const float m = warp_reduce(thread_max<D>(vv), [](float a, float b) { return max_nan(a, b); });
            best = merge_argmax(best, make_int2(__float_as_int(m), tile));
        }
        if (lane == 0) s_best[warp] = best;
        __syncthreads();
        if (tid == 0) {
            int2 b = s_best[0];
            for (int w = 1; w < kLzWarps; ++w) b = merge_argmax(b, s_best[w]);
            s_cbest[0] = b.x;
            s_cbest[1] = b.y;
        }
        csync<CS>();  // every CTA's best is written
        int2 b = make_int2(s_cbest[0], s_cbest[1]);
        if constexpr (CS > 1) {
            b = make_int2(ld_dsmem(dsmem_addr(&s_cbest[0], 0)), ld_dsmem(dsmem_addr(&s_cbest[1], 0)));
            for (int r = 1; r < CS; ++r)
                b = merge_argmax(b, make_int2(ld_dsmem(dsmem_addr(&s_cbest[0], r)), ld_dsmem(dsmem_addr(&s_cbest[1], r))));
        }
        const float bm = __int_as_float(b.x);
        const int tile = bm != bm ? -1 : b.y;
        // the first position of the maximum inside that tile, by the warp that read it
        const bool owner = tile >= 0 && (tile % (CS * kLzWarps)) == gwarp;
        if (owner) {
            const int64_t c0 = int64_t(tile) * TE;
            const int len = unit_len(V, c0, TE);
            if (held != tile) {
#pragma unroll
                for (int u = 0; u < kTileVecs; ++u) {
                    const int e0 = (lane + 32 * u) * D::EPV;
                    vv[u] = e0 < len ? load_vec<D, VEC>(row, c0, e0, len) : neg_inf_vec<D>();
                }
            }
            int idx = kNoIndex;
#pragma unroll
            for (int u = kTileVecs - 1; u >= 0; --u) {
                const int e0 = (lane + 32 * u) * D::EPV;
#pragma unroll
                for (int e = D::EPV - 1; e >= 0; --e) {
                    const bool hit = vec_elem<D>(vv[u], e) == bm && e0 + e < len;
                    idx = hit ? int(c0) + e0 + e : idx;
                }
            }
            idx = warp_reduce(idx, [](int a, int c) { return min(a, c); });
            if (lane == 0) s_idx = idx;
        }
        csync<CS>();  // the index is written (and every CTA is done reading the bests)
        int r = -1;
        if (tile >= 0) {
            const int orank = (tile % (CS * kLzWarps)) / kLzWarps;
            if constexpr (CS > 1) r = ld_dsmem(dsmem_addr(&s_idx, orank));
            else r = s_idx;
        }
        return r;
    };

    // accepted nodes in index order: their rows decide their children and the bonus
    int best = 0;
    for (int v = 0; v < N; ++v) {
        if (!s_acc[v]) continue;  // uniform: written before the last barrier
        const int a = row_argmax(v);
        if (a < 0) {  // a NaN in a row the rule reads
            csync<CS>();  // no CTA leaves while another may still read its shared memory
            fail();
            return;
        }
        if (tid == 0) s_arg[v] = a;
        for (int c = v + 1 + tid; c < N; c += kLzThreads)
            if (s_par[c] == v && s_tok[c] == a) s_acc[c] = 1;
        if (s_dep[v] > s_dep[best]) best = v;
        __syncthreads();
    }
    csync<CS>();  // the last index read of the cluster is done
    if (!writer) return;
    // outputs: the path root .. best, its tokens, the bonus argmax(best), -1 padding
    const int depth = s_dep[best];
    if (!SV_IN(depth, W)) return;
    if (tid == 0)
        for (int s = depth, node = best; s >= 0 && SV_IN(node, N); --s) {
            s_path[s] = node;
            node = s_par[node];
        }
    __syncthreads();
    for (int i = tid; i < W; i += kLzThreads) {
        if (opath) opath[i] = i <= depth ? s_path[i] : -1;
        out[i] = i < depth ? (SV_IN(s_path[i + 1], N) ? s_tok[s_path[i + 1]] : -1) : (i == depth ? s_arg[best] : -1);
    }
    if (tid == 0) accepted_len[seq] = depth;
}

template <int CS>
cudaError_t launch_walk_cs(int dtype, bool vec, Logits t, int B, int N, int V, bool chain, const int32_t *parent,
                           const int32_t *tokens, int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                           int32_t *out_path, size_t smem, cudaStream_t s) {
    auto k = dtype == 1 ? (vec ? greedy_walk_kernel<BF16, true, CS> : greedy_walk_kernel<BF16, false, CS>)
                        : (vec ? greedy_walk_kernel<F32, true, CS> : greedy_walk_kernel<F32, false, CS>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B) * CS);
    cfg.blockDim = dim3(kLzThreads);
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
    return cudaLaunchKernelEx(&cfg, k, t, N, V, chain, parent, tokens, max_depth, accepted_len, out_tokens, out_path);
}

cudaError_t launch_greedy_walk(int dtype, bool vec, Logits t, int B, int N, int V, bool chain, const int32_t *parent,
                               const int32_t *tokens, int max_depth, int32_t *accepted_len, int32_t *out_tokens,
                               int32_t *out_path, cudaStream_t s) {
    const size_t smem = size_t(5 * N + max_depth + 1) * sizeof(int);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // CTAs per sequence: the most (a power of two, at most 8) that still fit one wave
    int cs = 1;
    while (cs < 8 && int64_t(B) * cs * 2 <= sms) cs *= 2;
    switch (cs) {
    case 8: return launch_walk_cs<8>(dtype, vec, t, B, N, V, chain, parent, tokens, max_depth, accepted_len, out_tokens, out_path, smem, s);
    case 4: return launch_walk_cs<4>(dtype, vec, t, B, N, V, chain, parent, tokens, max_depth, accepted_len, out_tokens, out_path, smem, s);
    case 2: return launch_walk_cs<2>(dtype, vec, t, B, N, V, chain, parent, tokens, max_depth, accepted_len, out_tokens, out_path, smem, s);
    default: return launch_walk_cs<1>(dtype, vec, t, B, N, V, chain, parent, tokens, max_depth, accepted_len, out_tokens, out_path, smem, s);
    }
}

}  // namespace sv
