// sv_grid.cuh -- bounded device-side waits: a flag set by another warp of the grid, and a
// grid-wide barrier for cooperative launches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

constexpr uint64_t kBarrierLimitNs = 2000000000ull;  // give up a grid barrier after 2 s

// Control words of a grid barrier inside an int32 control block.
constexpr int kBarCount = 1, kBarGen = 2, kBarStatus = 3;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A load with acquire semantics at device scope (sees what a release -- a fence then a
// store or atomic -- made visible before it).
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Waits until *p is nonzero and returns it.  Gives up after limit_ns: records
// SV_ERR_TIMEOUT in *status and returns 0.  Only for flags that a warp already running
// (never itself waiting) will set.
__device__ inline int wait_nonzero(const int *p, int *status, uint64_t limit_ns) {
    int v = ld_acquire(p);
    if (v) return v;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        __nanosleep(128);
        v = ld_acquire(p);
        if (v) return v;
        if ((i & 15) == 15 && global_ns() - t0 > limit_ns) {
            atomicExch(status, int(SV_ERR_TIMEOUT));
            return 0;
        }
    }
}

// Grid barrier for a cooperative launch (all CTAs resident): waits until `expected` CTAs
// (the grid by default) have arrived.  ctl[kBarCount] must be 0 before the first barrier of
// a launch (the generation word may hold anything).  Returns false, after recording
// SV_ERR_TIMEOUT in ctl[kBarStatus], if the others did not arrive within limit_ns.
__device__ inline bool grid_barrier(int *ctl, int expected = -1, uint64_t limit_ns = kBarrierLimitNs) {
    if (expected < 0) expected = int(gridDim.x);
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int *gen = ctl + kBarGen;
        const int g = *gen;
        int ok = 1;
        __threadfence();
        if (atomicAdd(ctl + kBarCount, 1) == expected - 1) {
            atomicExch(ctl + kBarCount, 0);
            __threadfence();
            atomicAdd(ctl + kBarGen, 1);
        } else {
            const uint64_t t0 = global_ns();
            for (uint32_t i = 0; *gen == g; ++i) {
                if ((i & 63) == 63 && global_ns() - t0 > limit_ns) {
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        if (!ok) atomicExch(ctl + kBarStatus, int(SV_ERR_TIMEOUT));
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

// Arrival at a grid_barrier without the wait, for a CTA that leaves the kernel after it:
// the barrier's other CTAs still count it among the `expected` (the grid by default).
__device__ inline void grid_arrive(int *ctl, int expected = -1) {
    if (expected < 0) expected = int(gridDim.x);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(ctl + kBarCount, 1) == expected - 1) {
            atomicExch(ctl + kBarCount, 0);
            __threadfence();
            atomicAdd(ctl + kBarGen, 1);
        }
    }
}

}  // namespace sv
