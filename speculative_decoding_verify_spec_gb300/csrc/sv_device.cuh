// sv_device.cuh -- device-side building blocks of libspecverify (sm_103a).
//
// Unit of streaming work ("tile"): one warp covers kTileVecs 16-byte vectors per lane of
// one logits row, i.e. 4 KB (2048 bf16 or 1024 fp32 logits); lane l holds vectors
// l, l + 32, ... so every load instruction of the warp reads 512 contiguous bytes.  The
// streaming kernels are persistent: a grid of (SMs x resident CTAs) whose warps step through
// the tiles of all rows, each warp on its own, and write one partial per tile.
// A residual tile covers kResVecs vectors per lane of the target row and the same span of
// the draft row (2 KB of each).  In the in-order scan of the sampler lane l holds a
// contiguous run of vectors instead, so a per-lane prefix followed by a warp scan is in
// index order.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace sv {

constexpr int kThreads = 256;                          // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kTileVecs = 8;                           // 16-byte vectors per lane per tile
constexpr int kResVecs = 4;                            // ... per residual tile, of each row
constexpr int kNoIndex = 0x7FFFFFFF;                   // "no element" in argmax partials

// Element types.  EPV = elements per 16-byte vector; kNegInfWord = a 32-bit word whose
// elements are all -inf (the fill value of padding lanes).
struct F32 {
    static constexpr int EPV = 4;
    static constexpr int kBytes = 4;
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
};
struct BF16 {
    static constexpr int EPV = 8;
    static constexpr int kBytes = 2;
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
};

template <class D>
__host__ __device__ constexpr int tile_elems() { return 32 * kTileVecs * D::EPV; }
template <class D>
__host__ __device__ constexpr int res_tile_elems() { return 32 * kResVecs * D::EPV; }

// Number of real elements in the unit of `unit` elements that starts at element c0.
__device__ __forceinline__ int unit_len(int V, int64_t c0, int unit) {
    const int64_t rest = int64_t(V) - c0;
    return rest < unit ? int(rest) : unit;
}

// ------------------------------------------------------------------------------------
// Scalar helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {  // MUFU.EX2 (PTX ex2.approx.ftz.f32)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max_nan(float a, float b) {  // NaN-propagating max
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

__device__ __forceinline__ bool is_finite(float x) { return fabsf(x) < __int_as_float(0x7f800000); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Element j of a row (any alignment), widened to fp32.
template <class D>
__device__ __forceinline__ float load_elem(const char *row, int64_t j);
template <>
__device__ __forceinline__ float load_elem<F32>(const char *row, int64_t j) {
    return __ldg(reinterpret_cast<const float *>(row) + j);
}
template <>
__device__ __forceinline__ float load_elem<BF16>(const char *row, int64_t j) {
    return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short *>(row) + j)) << 16);
}

// Element e (0 <= e < EPV) of a packed vector, widened to fp32.
template <class D>
__device__ __forceinline__ float vec_elem(const uint4 &v, int e);
template <>
__device__ __forceinline__ float vec_elem<F32>(const uint4 &v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
}
template <>
__device__ __forceinline__ float vec_elem<BF16>(const uint4 &v, int e) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return (e & 1) ? bf16_hi(w) : bf16_lo(w);
}

// A 16-byte read-only load that is not kept in L1 and asks L2 to fetch the surrounding
// 256 bytes: logits are read once, in long runs.
__device__ __forceinline__ uint4 ld_stream(const char *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <class D>
__device__ __forceinline__ uint4 neg_inf_vec() {
    return make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
}

// ------------------------------------------------------------------------------------
// Loading one 16-byte vector of a unit (tile).  `e0` is the element offset of the vector
// inside the unit that starts at element c0, `len` the number of real elements in it.  A whole in-range vector of
// an aligned row is one 128-bit read-only load; anything else is read element by element
// and the missing elements are filled with -inf.
// ------------------------------------------------------------------------------------
template <class D, bool VEC>
__device__ __forceinline__ uint4 load_vec(const char *row, int64_t c0, int e0, int len) {
    if (VEC && e0 + D::EPV <= len) return ld_stream(row + (c0 + e0) * D::kBytes);
    uint32_t w[4] = {D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord};
    if constexpr (D::EPV == 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e0 + e < len) w[e] = __float_as_uint(load_elem<F32>(row, c0 + e0 + e));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e0 + e < len) {
                const uint32_t h = __float_as_uint(load_elem<BF16>(row, c0 + e0 + e)) >> 16;
                w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000FFFFu) | (h << 16))
                                    : ((w[e >> 1] & 0xFFFF0000u) | h);
            }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// NaN-propagating max over a packed vector.
template <class D>
__device__ __forceinline__ uint32_t vec_max_word(const uint4 &v);
template <>
__device__ __forceinline__ uint32_t vec_max_word<BF16>(const uint4 &v) {
    // max.NaN.bf16x2 on pairs: 3 ops for 8 elements
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162 *>(&v.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162 *>(&v.w);
    __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return *reinterpret_cast<uint32_t *>(&m);
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t x, uint32_t y) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&y);
    __nv_bfloat162 m = __hmax2_nan(a, b);
    return *reinterpret_cast<uint32_t *>(&m);
}

// Max (NaN-propagating) over a lane's N vectors, as fp32.
template <class D, int N>
__device__ __forceinline__ float thread_max(const uint4 (&v)[N]) {
    if constexpr (D::EPV == 8) {
        uint32_t m = vec_max_word<BF16>(v[0]);
#pragma unroll
        for (int u = 1; u < N; ++u) m = bf16x2_max_nan(m, vec_max_word<BF16>(v[u]));
        return max_nan(bf16_lo(m), bf16_hi(m));
    } else {
        float m = __uint_as_float(v[0].x);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            m = max_nan(m, __uint_as_float(v[u].x));
            m = max_nan(m, __uint_as_float(v[u].y));
            m = max_nan(m, __uint_as_float(v[u].z));
            m = max_nan(m, __uint_as_float(v[u].w));
        }
        return m;
    }
}

// sum_j 2^((x_j - m) c) over a thread's vectors.  x_j - m is exact for bf16 inputs (and
// within half an ulp for fp32), so each exponent carries a single rounding proportional to
// its own size -- the elements near the maximum, which carry the mass, are the most
// accurate.  Per pair of elements: one FADD2, one FMUL2, two MUFU.EX2, one FADD2.
template <class D, int N>
__device__ __forceinline__ float thread_sumexp(const uint4 (&v)[N], float c, float m) {
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
#pragma unroll
    for (int u = 0; u < N; ++u) {
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
            float2 a, b;
            if constexpr (D::EPV == 8) {
                a = make_float2(bf16_lo(w[q]), bf16_hi(w[q]));
                b = make_float2(bf16_lo(w[q + 1]), bf16_hi(w[q + 1]));
            } else {
                a = make_float2(__uint_as_float(w[q]), __uint_as_float(w[q + 1]));
                b = make_float2(0.f, 0.f);
            }
            const float2 ya = __fmul2_rn(__fadd2_rn(a, nm), cc);
            acc0 = __fadd2_rn(acc0, make_float2(ex2(ya.x), ex2(ya.y)));
            if constexpr (D::EPV == 8) {
                const float2 yb = __fmul2_rn(__fadd2_rn(b, nm), cc);
                acc1 = __fadd2_rn(acc1, make_float2(ex2(yb.x), ex2(yb.y)));
            }
        }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
}

// ------------------------------------------------------------------------------------
// Softmax statistics in base 2.  A partial (M, S) of a set of logits means
// S = sum 2^((l - M) c) with M the largest logit; M = NaN or +inf marks bad data,
// M = -inf an all -inf set (S = 0).
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float2 merge_stats(float2 a, float2 b, float c) {
    const float M = max_nan(a.x, b.x);
    if (!is_finite(M)) return make_float2(M, 0.f);
    const float S = a.y * ex2((a.x - M) * c) + b.y * ex2((b.x - M) * c);
    return make_float2(M, S);
}

// Argmax partial (value, index): larger value wins, equal values go to the lower index;
// a NaN value marks bad data and absorbs everything.
__device__ __forceinline__ int2 merge_argmax(int2 a, int2 b) {
    const float va = __int_as_float(a.x), vb = __int_as_float(b.x);
    if (va != va) return a;
    if (vb != vb) return b;
    if (vb > va || (vb == va && b.y < a.y)) return b;
    return a;
}

template <class T, class Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        T w;
        if constexpr (sizeof(T) == 8) {
            long long bits = *reinterpret_cast<long long *>(&v);
            bits = __shfl_xor_sync(0xFFFFFFFFu, bits, o);
            w = *reinterpret_cast<T *>(&bits);
        } else {
            w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        }
        v = op(v, w);
    }
    return v;
}

// Block-wide reduction over a CTA of NW warps; every thread returns the result.
// `scratch` holds NW values.
template <int NW, class T, class Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_reduce(v, op);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    T r = scratch[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) r = op(r, scratch[w]);
    return r;
}

// Inclusive scan of one float per lane across the warp (index order = lane order).
__device__ __forceinline__ float warp_inclusive_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float w = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += w;
    }
    return v;
}

// Compensated (Kahan) running sum, for the draw's prefixes: the threshold is compared with
// running sums of thousands of terms, where plain fp32 accumulation drifts.
struct Kahan {
    float sum = 0.f, comp = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float y = __fsub_rn(x, comp);
        const float t = __fadd_rn(sum, y);
        comp = __fsub_rn(__fsub_rn(t, sum), y);
        sum = t;
    }
    __device__ __forceinline__ float value() const { return __fsub_rn(sum, comp); }
};

// A warp's walk over the tiles of a persistent kernel: item it = (seq * R + local) * ntile
// + tile, stepped by the total number of warps without divisions after the first.
struct TileWalk {
    int64_t it, seq;
    int local, tile;
    int64_t step_seq;
    int step_local, step_tile;
    int R, ntile;
    __device__ TileWalk(int64_t it0, int64_t nwarps, int R_, int ntile_) : it(it0), R(R_), ntile(ntile_) {
        const int64_t row = it0 / ntile;
        tile = int(it0 - row * ntile);
        seq = row / R;
        local = int(row - seq * R);
        const int64_t dq = nwarps / ntile;
        step_tile = int(nwarps - dq * ntile);
        step_seq = dq / R;
        step_local = int(dq - step_seq * R);
    }
    __device__ void next(int64_t nwarps) {
        it += nwarps;
        tile += step_tile;
        int carry = 0;
        if (tile >= ntile) {
            tile -= ntile;
            carry = 1;
        }
        local += step_local + carry;
        seq += step_seq;
        if (local >= R) {
            local -= R;
            ++seq;
        }
    }
};

// Programmatic dependent launch.  Every kernel of a call first lets the next kernel of the
// call be scheduled (its CTAs then wait in griddep_wait on SMs freed by this grid's tail),
// then, before it reads anything an earlier kernel wrote, waits for the previous grid to
// complete and flush.  A call's first kernel waits before any read at all (its predecessor
// is the caller's kernel, which may signal its dependents before it has written the
// logits), so across calls only the launch latency is hidden.  Every CTA waits before it may exit, so a grid is only complete once
// its predecessor is -- completion is transitive along the call.  For a grid launched
// without the attribute both instructions are no-ops.
__device__ __forceinline__ void griddep_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// All threads of a thread-block cluster of CS CTAs (CS = 1: the CTA).  The .release /
// .acquire barrier orders the threads' memory operations at cluster scope, so what one CTA
// wrote before it (shared or global) is seen after it by the others.
template <int CS>
__device__ __forceinline__ void csync() {
    if constexpr (CS > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
        __syncthreads();
    }
}
template <int CS>
__device__ __forceinline__ int cluster_rank() {
    if constexpr (CS > 1) {
        unsigned r;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
        return int(r);
    } else {
        return 0;
    }
}

// Distributed shared memory: the address of this CTA's shared variable *p in the shared
// memory of cluster CTA `rank`, and 32-bit loads from such an address.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
    return r;
}
__device__ __forceinline__ int ld_dsmem(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Launches `kernel` so that it may start while the previous kernel on the stream drains;
// a cooperative launch (every CTA resident at once) when asked.
template <class... Params, class... Args>
inline cudaError_t launch_after_ex(bool cooperative, void (*kernel)(Params...), unsigned grid, unsigned block,
                                   size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cooperative ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
template <class... Params, class... Args>
inline cudaError_t launch_after(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                                cudaStream_t s, Args &&...args) {
    return launch_after_ex(false, kernel, grid, block, smem, s, std::forward<Args>(args)...);
}

// One warp merges the n tile partials of a row: lane l takes tiles l, l + 32, ... in order,
// then the lanes combine in a fixed butterfly.  Every lane returns the row's result.  L2:
// read the partials at L2 (written by other SMs in the same kernel, after a fence).
template <bool L2 = false>
__device__ __forceinline__ float2 warp_merge_stats(const float2 *__restrict__ p, int n, float c, int lane) {
    float2 s = make_float2(-__int_as_float(0x7f800000), 0.f);
    for (int q0 = lane; q0 < n; q0 += 128) {
        float2 e[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            e[j] = q0 + 32 * j < n ? (L2 ? __ldcg(p + q0 + 32 * j) : p[q0 + 32 * j])
                                   : make_float2(-__int_as_float(0x7f800000), 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) s = merge_stats(s, e[j], c);
    }
    return warp_reduce(s, [c](float2 a, float2 b) { return merge_stats(a, b, c); });
}
__device__ __forceinline__ int2 warp_merge_argmax(const int2 *__restrict__ p, int n, int lane) {
    int2 s = make_int2(__float_as_int(-__int_as_float(0x7f800000)), kNoIndex);
    for (int q0 = lane; q0 < n; q0 += 128) {
        int2 e[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            e[j] = q0 + 32 * j < n ? p[q0 + 32 * j] : make_int2(__float_as_int(-__int_as_float(0x7f800000)), kNoIndex);
#pragma unroll
        for (int j = 0; j < 4; ++j) s = merge_argmax(s, e[j]);
    }
    return warp_reduce(s, [](int2 a, int2 b) { return merge_argmax(a, b); });
}

// The persistent streaming grid: SMs x resident CTAs of `kernel`, at most enough CTAs to
// give every warp one of `items` tiles.
template <class K>
inline cudaError_t persistent_grid(K kernel, int64_t items, unsigned *grid) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t need = (items + kWarps - 1) / kWarps;
    const int64_t full = int64_t(sms) * per_sm;
    *grid = unsigned(need < full ? (need > 0 ? need : 1) : full);
    return cudaSuccess;
}

// ------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): ten rounds; round r uses the key plus r times the
// Weyl increments (0x9E3779B9, 0xBB67AE85); multipliers 0xD2511F53 and 0xCD9E8D57.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint2 key) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_hi = __umulhi(0xD2511F53u, ctr.x), a_lo = 0xD2511F53u * ctr.x;
        const uint32_t b_hi = __umulhi(0xCD9E8D57u, ctr.z), b_lo = 0xCD9E8D57u * ctr.z;
        ctr = make_uint4(b_hi ^ ctr.y ^ key.x, b_lo, a_hi ^ ctr.w ^ key.y, a_lo);
        key.x += 0x9E3779B9u;
        key.y += 0xBB67AE85u;
    }
    return ctr;
}

// The verifier's uniform at (sequence b, position i, purpose): word 0 of Philox at counter
// (4 i + purpose, b, offset lo, offset hi), key (seed lo, seed hi); (w >> 8) * 2^-24.
__device__ __forceinline__ float uniform01(uint64_t seed, uint64_t offset, uint32_t b, uint32_t i,
                                           uint32_t purpose) {
    const uint4 ctr = make_uint4((i << 2) | (purpose & 3u), b, uint32_t(offset), uint32_t(offset >> 32));
    const uint2 key = make_uint2(uint32_t(seed), uint32_t(seed >> 32));
    return float(philox4x32_10(ctr, key).x >> 8) * 0x1p-24f;
}

}  // namespace sv
