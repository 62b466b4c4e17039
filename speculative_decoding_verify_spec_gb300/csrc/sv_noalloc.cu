// sv_noalloc.cu -- greedy verification for callers that cannot allocate device memory.
//
// spec_verify_greedy needs a caller-provided workspace for its per-tile maxima.
// Some callers have no way to provide one: code that runs inside another runtime's
// execution step (a plugin or custom op whose host framework owns every device buffer and
// forbids allocation while a request is in flight), or a serving loop that must never call
// cudaMalloc after start-up because it can block on other streams and fragments a fixed
// memory budget.  For them this file keeps its scratch in a fixed device array that is
// part of the loaded library image, so the call allocates nothing at all.
//
// The array is kNoallocScratchBytes (SV_NOALLOC_SCRATCH_BYTES) long, 256-byte aligned, and
// every GPU that loads the library holds one copy until the process exits.  All calls on a
// device share it: nothing in it needs clearing between calls (every partial is written
// before it is read), but two calls whose kernels overlap on the GPU -- e.g. on different
// streams -- race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "spec_verify.h"
#include "sv_device.cuh"
#include "sv_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = SV_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_greedy_scratch[kNoallocScratchBytes];

// The array's device address, looked up once per device.  In host code the name
// g_greedy_scratch is only a host-side handle, never a usable device pointer.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_lock;

sv_status scratch_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_scratch_lock);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_greedy_scratch) != cudaSuccess || p == nullptr)
            return SV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_greedy_noalloc(const void *target_logits, int64_t t_batch_stride,
                                                int64_t t_row_stride, sv_dtype dtype, int B,
                                                int gamma, int V, const int32_t *draft_tokens,
                                                int32_t *accepted_len, int32_t *out_tokens,
                                                void *stream) {
    if (dtype != SV_FP32 && dtype != SV_BF16) return SV_ERR_UNSUPPORTED;
    if (B < 0 || gamma < 0 || gamma > SV_MAX_GAMMA || V < 1 || V > SV_MAX_VOCAB)
        return SV_ERR_INVALID_ARG;
    if (t_batch_stride < 0 || t_row_stride < 0) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !accepted_len || !out_tokens || (gamma > 0 && !draft_tokens))
        return SV_ERR_INVALID_ARG;
    const int ntile = sv::ntile_of(V, dtype);
    const int64_t partials = int64_t(B) * (gamma + 1) * ntile;
    if (partials * int64_t(sizeof(float)) > int64_t(kNoallocScratchBytes))
        return SV_ERR_WORKSPACE;  // larger than the fixed scratch: use spec_verify_greedy
    void *scratch = nullptr;
    if (sv_status st = scratch_address(&scratch)) return st;
    const bool vec = sv::vec_ok(target_logits, t_batch_stride, t_row_stride, dtype);
    const sv::Logits t{target_logits, t_batch_stride, t_row_stride};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = sv::mark_stage(0, s);  // the same stage events as spec_verify_greedy
    if (e == cudaSuccess) e = sv::launch_max_tiles(dtype == SV_BF16, vec, t, gamma + 1, B, V, ntile, scratch, s);
    if (e == cudaSuccess) e = sv::mark_stage(1, s);
    if (e == cudaSuccess)
        e = sv::launch_greedy_finalize(dtype == SV_BF16, vec, t, B, gamma, V, ntile, scratch, draft_tokens,
                                       accepted_len, out_tokens, s);
    if (e == cudaSuccess) e = sv::mark_stage(2, s);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
