// Pieces shared by the FP8 and BF16 attention kernels: kernel parameters,
// the bounded mbarrier wait, register pinning after TMEM loads, 2^k.
#pragma once

#include <cstdint>

#include "checked.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

constexpr long long ATTN_WAIT_LIMIT = 1000000000LL;  // cycles (~0.5 s) before a wait gives up

struct AttnParams {
    const int32_t* cu;
    const int32_t* order;
    const int32_t* prefix;
    WsHeader* ws;
    const vitfp8_scale_state* st;
    uint16_t* out;
    int nseq, T, H, D, Dp, DV, KS;
    float sm_scale;
    int64_t out_elems;  // T * H * D (checked build)
};

// Bounded wait: true when the phase with `parity` completed; false if the CTA
// aborted or this wait timed out (which sets the abort flag and the error).
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      int32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((it & 7u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > ATTN_WAIT_LIMIT) {
                *abort_flag = 1;
                record_error(err, VITFP8_ERR_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

// 2^k for an integer-valued float k in [-126, 0].
__device__ __forceinline__ float exp2_int(float k) {
    int e = int(k) + 127;
    e = e < 1 ? 1 : e;
    return __int_as_float(e << 23);
}

}  // namespace vitfp8
