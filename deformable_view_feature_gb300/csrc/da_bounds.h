// Index checks of the bounds-checking build (DA_DEBUG_BOUNDS).
//
// da_index_ok(i, n) is the predicate every checked access goes through: it
// holds exactly when 0 <= i < n. Plain C++ (host and device), so the host
// tests compile it on its own. In a kernel, DA_CHECK(err, i, n, bit) is
// that predicate in a bounds-checking build, setting `bit` in the device
// error word *err when it fails (the caller then skips the access); in a
// release build it is the constant true and costs nothing.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DA_HD __host__ __device__
#else
#define DA_HD
#endif

namespace da {

DA_HD inline bool da_index_ok(int64_t i, int64_t n) { return i >= 0 && i < n; }

// Kinds of checked index: one bit each in the error word.
enum : uint32_t {
    kBoundsFeatRow = 1u << 0,   // feature / grad_feat row from a sampling location
    kBoundsOutput = 1u << 1,    // element of out, grad_loc, grad_weight and the like
    kBoundsRecord = 1u << 2,    // record slot of the binned backward
    kBoundsAnchor = 1u << 3,    // anchor decoded from a record
    kBoundsSample = 1u << 4,    // sample id decoded from a record (weights, d)
    kBoundsRowCount = 1u << 5,  // per-row counter or offset of the binning
    kBoundsShared = 1u << 6,    // shared-memory table entry
    kBoundsPixel = 1u << 7,     // source pixel of the warpaffine kernels
};

}  // namespace da

#if defined(__CUDACC__)
#ifdef DA_DEBUG_BOUNDS
namespace da {
__device__ __forceinline__ bool da_check_dev(uint32_t *err, int64_t i, int64_t n, uint32_t bit)
{
    if (da_index_ok(i, n)) return true;
    if (err) atomicOr(err, bit);
    return false;
}
}  // namespace da
#define DA_CHECK(err, i, n, bit) ::da::da_check_dev((err), static_cast<int64_t>(i), static_cast<int64_t>(n), (bit))
#else
#define DA_CHECK(err, i, n, bit) true
#endif
#endif
