// sv_checks.cuh -- the bounds-checked build of the library (compiled with -DSV_CHECKS).
//
// The library knows the extent of every buffer it indexes on its own: the workspace regions
// it lays out (tile partials B x R x ntile, row statistics B x R, plans B, residual masses
// B x nrt, re-draw records 2 B, unit sums, level lists ...), the tile and unit counts of a
// row, the tree's node ids (0 .. N - 1), and the caller's outputs (B, B x (gamma + 1)).  In
// the checked build every such index goes through SV_IN(index, extent) before the access:
// an index outside [0, extent) records the first violation -- the site (a tag of the source
// file and the line), the index and the extent -- in a device error word, and the access
// is skipped (a load yields a neutral value).  spec_verify_check_word() returns that word
// to the host and clears it.  In the normal build SV_IN is the constant true and costs
// nothing.
#pragma once

#include <stdint.h>

namespace sv {

// A 16-bit tag of a source file's base name (FNV-1a over the characters after the last
// '/', folded to 16 bits), computed at compile time.
__host__ __device__ constexpr const char *base_name(const char *s, const char *b) {
    return *s ? base_name(s + 1, *s == '/' ? s + 1 : b) : b;
}
__host__ __device__ constexpr uint32_t fnv_tag(const char *s, uint32_t h = 2166136261u) {
    return *s ? fnv_tag(s + 1, (h ^ uint32_t(uint8_t(*s))) * 16777619u) : ((h >> 16) ^ (h & 0xFFFFu));
}
__host__ __device__ constexpr uint32_t file_tag(const char *path) { return fnv_tag(base_name(path, path)); }
template <uint32_t T>
struct SiteTag {
    static constexpr uint32_t value = T;
};

#ifdef SV_CHECKS
// [0] site of the first violation (file tag << 16 | line; 0: none), [1] the index (clamped
// to int32), [2] the extent (clamped), [3] violations seen.
extern __device__ int g_check[4];
__device__ bool check_fail(uint32_t site, int64_t idx, int64_t n);
#define SV_IN(idx, n)                                                                            \
    ((int64_t(idx) >= 0 && int64_t(idx) < int64_t(n))                                           \
         ? true                                                                                  \
         : ::sv::check_fail((::sv::SiteTag<::sv::file_tag(__FILE__)>::value << 16) | uint32_t(__LINE__), \
                            int64_t(idx), int64_t(n)))
#else
#define SV_IN(idx, n) true
#endif

}  // namespace sv
