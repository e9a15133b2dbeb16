// Internal declarations shared by the host API (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "vitfp8.h"

namespace vitfp8 {

// Source layout as passed to kernels (by value).
struct SrcDev {
    int32_t padded;
    int64_t s_max;
    int64_t ts;  // token stride, elements
    int64_t hs;  // head stride, elements
    int64_t extent;  // elements the layout addresses (checked build)
};

// Attention workspace: a header, then one record per segment in the work
// list's order (longest first), so that a CTA finds its segment with one
// 16-byte load per probe; then the key-range split's arrival counters and
// partial results (FP8 kernel only).
struct WsHeader {
    int32_t error;        // first device-detected vitfp8_status
    int32_t total_items;  // work items of the current call
    int32_t num_seqs;
    int32_t split_first;  // first work item whose key range is split (total_items: none)
    int32_t split_k;      // parts per split item (1: none)
    int32_t next_unit;    // FP8 kernel: units handed out beyond the first wave (zeroed by the plan)
    int32_t pad[10];
};
static_assert(sizeof(WsHeader) == 64, "workspace header is 64 bytes");

struct SegRec {
    int32_t first_item;   // work items of all earlier records
    int32_t seg_s, seg_e; // the segment's packed token range
    int32_t nq;           // its query tiles (items per head)
};
static_assert(sizeof(SegRec) == 16, "one 16-byte load per record");

// Key-range split of the last, partly filled wave of work items: at most
// kSplitMaxParts CTAs (one wave) and kSplitMaxK parts per item; each part
// leaves kSplitPartBytes of partial results.
constexpr int kSplitMaxParts = 160;
constexpr int kSplitMaxK = 4;
constexpr size_t kSplitPartBytes = 84 * 1024;

constexpr size_t ws_rec_bytes(int32_t num_seqs) {
    return (sizeof(WsHeader) + sizeof(SegRec) * size_t(num_seqs) + 255) & ~size_t(255);
}
constexpr size_t ws_split_cnt_offset(int32_t num_seqs) { return ws_rec_bytes(num_seqs); }
constexpr size_t ws_split_part_offset(int32_t num_seqs) { return ws_rec_bytes(num_seqs) + 1024; }
static_assert(kSplitMaxParts * sizeof(int32_t) <= 1024, "split counters fit their block");
constexpr size_t ws_bytes(int32_t num_seqs) {
    return ws_split_part_offset(num_seqs) + size_t(kSplitMaxParts) * kSplitPartBytes;
}

__device__ __forceinline__ void record_error(int32_t* word, int32_t code) {
    atomicCAS(word, 0, code);
}

// ---- launchers (quant.cu)
cudaError_t launch_state_init(vitfp8_scale_state* st, cudaStream_t s);
cudaError_t launch_set_static(vitfp8_scale_state* st, float q, float k, float v, cudaStream_t s);
cudaError_t launch_amax(vitfp8_scale_state* st, const uint16_t* q, const uint16_t* k,
                        const uint16_t* v, SrcDev L, const int32_t* cu, int nseq, int T, int H,
                        int D, float* out, cudaStream_t s);
cudaError_t launch_ring_push(vitfp8_scale_state* st, const float* vals, cudaStream_t s);
cudaError_t launch_calibrated_scales(const vitfp8_scale_state* dyn, float margin, float* out,
                                     vitfp8_scale_state* dst, cudaStream_t s);
cudaError_t launch_set_ring_order(vitfp8_scale_state* st, int delayed, cudaStream_t s);
cudaError_t launch_quant(const vitfp8_scale_state* st, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, SrcDev L, const int32_t* cu, int nseq, int T, int H,
                         int D, int Dp, uint8_t* q8, uint8_t* k8, uint8_t* v8t, int64_t Tv,
                         cudaStream_t s);

// ---- launchers (selftest.cu)
cudaError_t launch_selftest_wait(void* ws, cudaStream_t s);
cudaError_t launch_selftest_bounds(void* ws, cudaStream_t s);

// ---- launchers (attn_fp8.cu)
// split_bn > 0 and nsm > 0 let the plan split the key ranges (tiles of
// split_bn keys) of the last wave's items over up to nsm CTAs.
cudaError_t launch_attn_plan(const int32_t* cu, int nseq, int T, int H, int rows_per_item,
                             int nsm, int split_bn, void* ws, cudaStream_t s);
// FP8 attention kernels (the values of vitfp8_attn_kernel in vitfp8.h).
constexpr int kAttnAuto = 0;        // attn_fp8_kernel_for() picks
constexpr int kAttnUnit = 1;        // one CTA per 128-row work item (attn_fp8.cu)
constexpr int kAttnPersistent = 2;  // one CTA per SM walking the work items (attn_fp8.cu)
constexpr int kAttnTwoTile = 3;     // one CTA per 256-row unit, two query tiles (attn_fp8_2tile.cu)
constexpr int kAttnTwoTilePersistent = 4;  // the two-tile units run by one CTA per SM
// Two-tile kernels: at least kTwoTileMinWaves waves of 256-row units; for
// segments of kTwoTileLongSeqlen tokens or more (where the two-tile kernels
// gain only a few per cent per unit) also the last wave's shortfall at most
// kTwoTileMaxTail of the time (ceil(w) / w <= 1 + kTwoTileMaxTail).
constexpr int kTwoTileLongSeqlen = 2048;
constexpr double kTwoTileMinWaves = 2.0;
constexpr double kTwoTileMaxTail = 0.12;
// Persistent kernels: longest segment at most this long (the one-tile one also
// needs more than one wave of items).
constexpr int kPersistentMaxSeqlen = 6144;

// The kernel the FP8 attention call runs when none is asked for, from what
// the host knows: segment count, the bound on segment lengths, token count,
// heads and SM count.  The two-tile kernels' units are estimated as
// H * (T + 128 * nseq) / 256 (a segment's last unit is half full on average).
inline int attn_fp8_kernel_for(int nseq, int max_seqlen, int T, int H, int nsm) {
    if (nsm <= 0 || nseq <= 0 || T <= 0 || H <= 0) return kAttnUnit;
    const double waves = double(H) * (double(T) + 128.0 * nseq) / 256.0 / double(nsm);
    if (waves >= kTwoTileMinWaves) {
        double full = double(int64_t(waves));
        if (full < waves) full += 1.0;
        if (max_seqlen < kTwoTileLongSeqlen || full <= waves * (1.0 + kTwoTileMaxTail))
            return max_seqlen <= kPersistentMaxSeqlen ? kAttnTwoTilePersistent : kAttnTwoTile;
    }
    const long long max_items = (long long)((T + 127) / 128 + nseq) * H;
    if (max_seqlen <= kPersistentMaxSeqlen && max_items > nsm) return kAttnPersistent;
    return kAttnUnit;
}

// kernel: one of the kAttn* values (kAttnAuto: attn_fp8_kernel_for).  All
// kernels compute the same attention; the unit and persistent kernels give
// the same bits, the two-tile kernel can differ in the last bit of about 1 %
// of the outputs (its reference moves at 128-key boundaries).
vitfp8_status launch_attn_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                              const vitfp8_scale_state* st, const int32_t* cu, int nseq, int max_seqlen,
                              int T, int H, int D, int Dp, int64_t Tv, float sm_scale, uint16_t* out,
                              void* ws, int kernel, cudaStream_t s);

// ---- launcher (attn_bf16.cu)
vitfp8_status launch_attn_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* cu, int nseq, int max_seqlen, int T, int H, int D,
                               float sm_scale, uint16_t* out, void* ws, cudaStream_t s);

}  // namespace vitfp8
