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
    const SegRec* rec;      // work-list records, longest segment first
    WsHeader* ws;
    const vitfp8_scale_state* st;
    uint16_t* out;
    int32_t* split_cnt;     // per split work item: parts finished (zeroed by the plan)
    float* split_part;      // per split part: kSplitPartBytes of partial results
    int nseq, T, H, D, Dp, DV, KS;
    float sm_scale;
    int64_t out_elems;  // T * H * D (checked build)
};

// The two-tile FP8 kernels (attn_fp8_2tile.cu): plan 256-row units and
// launch one CTA per unit or (persistent) one CTA per SM; the tensor maps are
// attn_fp8.cu's with a 128-key K box.
vitfp8_status launch_attn_fp8_2tile(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                    const AttnParams& prm, int nsm, bool persistent, cudaStream_t s);

// Work item -> the record of its segment (the last record whose first_item
// is <= item).  In two steps so that a caller can issue every load it needs
// before it knows the item: find_item_load reads, with at most 32 records,
// the calling lane's record (every lane of the warp must call both steps);
// find_item_pick then picks the record by a vote, or else binary-searches the
// records.  False (checked build) if an index falls outside the work list,
// or if item is past every record.
__device__ __forceinline__ int4 find_item_load(const AttnParams& p) {
    const int lane = threadIdx.x & 31;
    int4 mine = make_int4(0x7FFFFFFF, 0, 0, 0);
    if (p.nseq <= 32 && lane < p.nseq && VF_IN(lane, 1, p.nseq, &p.ws->error))
        mine = *reinterpret_cast<const int4*>(p.rec + lane);
    return mine;
}

__device__ __forceinline__ bool find_item_pick(const AttnParams& p, int item, int4 mine, SegRec& r) {
    const int lane = threadIdx.x & 31;
    if (p.nseq <= 32) {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, lane < p.nseq && mine.x <= item);
        if (m == 0u) return false;   // only when item is past every record (no work)
        const int lo = 31 - __clz(m);
        r.first_item = __shfl_sync(0xFFFFFFFFu, mine.x, lo);
        r.seg_s = __shfl_sync(0xFFFFFFFFu, mine.y, lo);
        r.seg_e = __shfl_sync(0xFFFFFFFFu, mine.z, lo);
        r.nq = __shfl_sync(0xFFFFFFFFu, mine.w, lo);
        return true;
    }
    int lo = 0, hi = p.nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (!VF_IN(mid, 1, p.nseq, &p.ws->error)) return false;
        if (p.rec[mid].first_item <= item) lo = mid; else hi = mid - 1;
    }
    if (!VF_IN(lo, 1, p.nseq, &p.ws->error)) return false;
    const int4 v = *reinterpret_cast<const int4*>(p.rec + lo);
    r.first_item = v.x;
    r.seg_s = v.y;
    r.seg_e = v.z;
    r.nq = v.w;
    return true;
}

// Both steps, and the call's item count.
__device__ __forceinline__ bool find_item(const AttnParams& p, int item, SegRec& r, int& total) {
    total = p.ws->total_items;
    return find_item_pick(p, item, find_item_load(p), r);
}

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
