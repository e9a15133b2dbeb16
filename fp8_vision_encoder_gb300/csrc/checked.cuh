// Checked build: compiled with -DVITFP8_CHECKED, every global- and shared-
// memory index the kernels compute is compared with the extent of its buffer
// before the access.  An index outside records VITFP8_ERR_DEVICE_BOUNDS in the
// launch's device error word and the access is skipped (a skipped load reads
// zeros); nothing traps or asserts, and the kernel runs to its end.  The same
// holds for the TMA rule that a copy's innermost coordinate be 16-byte
// aligned.  In the normal build every check compiles to `true` and costs
// nothing.
//
// Extents are those the arguments imply: a source tensor holds the rows its
// layout addresses, codes [T, H, D_pad] and [H, D_pad, Tv], the output
// [T, H, D], cu_seqlens num_seqs + 1 entries, the work list num_seqs and
// num_seqs + 1 entries.  The checks therefore catch a kernel that indexes
// outside what its arguments describe; the caller's allocations are guarded
// by the tests' canary bands.
#pragma once

#include <cstdint>

#include "internal.cuh"

namespace vitfp8 {

// [i, i + width) inside [0, n)?  Records the error if not.
__device__ __forceinline__ bool vf_in_range(int64_t i, int64_t width, int64_t n, int32_t* err) {
    if (i >= 0 && width >= 0 && i + width <= n) return true;
    record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
    return false;
}

}  // namespace vitfp8

#ifdef VITFP8_CHECKED
#define VF_IN(i, width, n, err) ::vitfp8::vf_in_range(int64_t(i), int64_t(width), int64_t(n), (err))
#define VF_CHECKED_BUILD 1
#else
#define VF_IN(i, width, n, err) true
#define VF_CHECKED_BUILD 0
#endif
