// Host side of the C ABI: argument validation and launches.  Every check runs
// before any launch; on failure nothing is enqueued.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "checked.cuh"
#include "internal.cuh"
#include "vitfp8.h"

using namespace vitfp8;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

vitfp8_status check_src(const vitfp8_src_layout* lay, int32_t H, int32_t D, SrcDev* out) {
    if (!lay) return VITFP8_ERR_INVALID_ARG;
    if (lay->padded != 0 && lay->padded != 1) return VITFP8_ERR_INVALID_ARG;
    if (lay->token_stride <= 0 || lay->head_stride < 0) return VITFP8_ERR_INVALID_ARG;
    if ((lay->token_stride & 7) || (lay->head_stride & 7)) return VITFP8_ERR_INVALID_ARG;
    if (H > 1 && lay->head_stride < D) return VITFP8_ERR_INVALID_ARG;
    if (lay->padded && lay->s_max <= 0) return VITFP8_ERR_INVALID_ARG;
    out->padded = lay->padded;
    out->s_max = lay->s_max;
    out->ts = lay->token_stride;
    out->hs = lay->head_stride;
    out->extent = 0;
    return VITFP8_OK;
}

// Elements a source tensor holds under its layout: the last addressed row's
// last head slice ends there (used by the checked build's bounds checks).
int64_t src_extent(const SrcDev& L, int32_t num_seqs, int32_t T, int32_t H, int32_t D) {
    const int64_t rows = L.padded ? int64_t(num_seqs) * L.s_max : int64_t(T);
    if (rows <= 0) return 0;
    return (rows - 1) * L.ts + int64_t(H - 1) * L.hs + D;
}

vitfp8_status check_common(const vitfp8_scale_state* st, const void* q, const void* k,
                           const void* v, const int32_t* cu, int32_t num_seqs, int32_t T,
                           int32_t H, int32_t D) {
    if (!st || !aligned4(st)) return VITFP8_ERR_INVALID_ARG;
    if (num_seqs < 0 || T < 0 || H <= 0) return VITFP8_ERR_INVALID_ARG;
    if (D < 8 || (D & 7)) return VITFP8_ERR_INVALID_ARG;
    if (D > 256) return VITFP8_ERR_UNSUPPORTED;
    if (num_seqs == 0 || T == 0) return VITFP8_OK;
    if (!q || !k || !v || !cu) return VITFP8_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned4(cu)) return VITFP8_ERR_INVALID_ARG;
    return VITFP8_OK;
}

}  // namespace

extern "C" {

const char* vitfp8_status_string(vitfp8_status s) {
    switch (s) {
        case VITFP8_OK: return "ok";
        case VITFP8_ERR_INVALID_ARG: return "invalid argument";
        case VITFP8_ERR_UNSUPPORTED: return "unsupported configuration";
        case VITFP8_ERR_CUDA: return "CUDA call failed";
        case VITFP8_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case VITFP8_ERR_DEVICE_BOUNDS: return "device index out of bounds";
        case VITFP8_ERR_BAD_SEQLENS: return "malformed cu_seqlens";
        case VITFP8_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int32_t vitfp8_version(void) { return 101; }

vitfp8_status vitfp8_scale_state_init(vitfp8_scale_state* d_state, cudaStream_t stream) {
    if (!d_state || !aligned4(d_state)) return VITFP8_ERR_INVALID_ARG;
    return launch_state_init(d_state, stream) == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_set_static_scales(vitfp8_scale_state* d_state, float q, float k, float v,
                                       cudaStream_t stream) {
    if (!d_state || !aligned4(d_state)) return VITFP8_ERR_INVALID_ARG;
    const float a[3] = {q, k, v};
    for (float x : a)
        if (!std::isfinite(x) || !(x > 0.0f)) return VITFP8_ERR_INVALID_ARG;
    return launch_set_static(d_state, q, k, v, stream) == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_amax_update(vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                 const vitfp8_bf16* k, const vitfp8_bf16* v,
                                 const vitfp8_src_layout* h_layout, const int32_t* d_cu_seqlens,
                                 int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t D,
                                 cudaStream_t stream) {
    vitfp8_status s = check_common(d_state, q, k, v, d_cu_seqlens, num_seqs, total_tokens, H, D);
    if (s != VITFP8_OK) return s;
    SrcDev L;
    s = check_src(h_layout, H, D, &L);
    if (s != VITFP8_OK) return s;
    L.extent = src_extent(L, num_seqs, total_tokens, H, D);
    if (num_seqs == 0 || total_tokens == 0) return VITFP8_OK;
    return launch_amax(d_state, q, k, v, L, d_cu_seqlens, num_seqs, total_tokens, H, D, nullptr,
                       stream) == cudaSuccess
               ? VITFP8_OK
               : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_amax_local(vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                const vitfp8_bf16* k, const vitfp8_bf16* v,
                                const vitfp8_src_layout* h_layout, const int32_t* d_cu_seqlens,
                                int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t D,
                                float* d_vals, cudaStream_t stream) {
    if (!d_vals || !aligned4(d_vals)) return VITFP8_ERR_INVALID_ARG;
    vitfp8_status s = check_common(d_state, q, k, v, d_cu_seqlens, num_seqs, total_tokens, H, D);
    if (s != VITFP8_OK) return s;
    SrcDev L;
    s = check_src(h_layout, H, D, &L);
    if (s != VITFP8_OK) return s;
    L.extent = src_extent(L, num_seqs, total_tokens, H, D);
    if (num_seqs == 0 || total_tokens == 0)
        return cudaMemsetAsync(d_vals, 0, 4 * sizeof(float), stream) == cudaSuccess ? VITFP8_OK
                                                                                    : VITFP8_ERR_CUDA;
    return launch_amax(d_state, q, k, v, L, d_cu_seqlens, num_seqs, total_tokens, H, D, d_vals,
                       stream) == cudaSuccess
               ? VITFP8_OK
               : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_set_ring_order(vitfp8_scale_state* d_state, int32_t delayed,
                                    cudaStream_t stream) {
    if (!d_state || !aligned4(d_state)) return VITFP8_ERR_INVALID_ARG;
    return launch_set_ring_order(d_state, delayed ? 1 : 0, stream) == cudaSuccess ? VITFP8_OK
                                                                                  : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_ring_push(vitfp8_scale_state* d_state, const float* d_vals,
                               cudaStream_t stream) {
    if (!d_state || !d_vals || !aligned4(d_state) || !aligned4(d_vals)) return VITFP8_ERR_INVALID_ARG;
    return launch_ring_push(d_state, d_vals, stream) == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_calibrated_scales(const vitfp8_scale_state* d_dynamic, float margin,
                                       float* d_saved, vitfp8_scale_state* d_static,
                                       cudaStream_t stream) {
    if (!d_dynamic || !aligned4(d_dynamic)) return VITFP8_ERR_INVALID_ARG;
    if (!std::isfinite(margin) || !(margin > 0.0f)) return VITFP8_ERR_INVALID_ARG;
    if (d_saved && !aligned4(d_saved)) return VITFP8_ERR_INVALID_ARG;
    if (d_static && !aligned4(d_static)) return VITFP8_ERR_INVALID_ARG;
    if (d_static == d_dynamic) return VITFP8_ERR_INVALID_ARG;
    return launch_calibrated_scales(d_dynamic, margin, d_saved, d_static, stream) == cudaSuccess
               ? VITFP8_OK
               : VITFP8_ERR_CUDA;
}

int64_t vitfp8_vt_stride(int32_t total_tokens) {
    if (total_tokens < 0) return 0;
    return (int64_t(total_tokens) + 15) & ~int64_t(15);
}

vitfp8_status vitfp8_quantize_unpad(const vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                    const vitfp8_bf16* k, const vitfp8_bf16* v,
                                    const vitfp8_src_layout* h_layout,
                                    const int32_t* d_cu_seqlens, int32_t num_seqs,
                                    int32_t total_tokens, int32_t H, int32_t D, int32_t D_pad,
                                    uint8_t* q8, uint8_t* k8, uint8_t* v8t, cudaStream_t stream) {
    vitfp8_status s = check_common(d_state, q, k, v, d_cu_seqlens, num_seqs, total_tokens, H, D);
    if (s != VITFP8_OK) return s;
    SrcDev L;
    s = check_src(h_layout, H, D, &L);
    if (s != VITFP8_OK) return s;
    L.extent = src_extent(L, num_seqs, total_tokens, H, D);
    if (D_pad < D || (D_pad & 15)) return VITFP8_ERR_INVALID_ARG;
    if (D_pad > 256) return VITFP8_ERR_UNSUPPORTED;
    if (num_seqs == 0 || total_tokens == 0) return VITFP8_OK;
    if (!q8 || !k8 || !v8t || !aligned16(q8) || !aligned16(k8) || !aligned16(v8t))
        return VITFP8_ERR_INVALID_ARG;
    return launch_quant(d_state, q, k, v, L, d_cu_seqlens, num_seqs, total_tokens, H, D, D_pad, q8,
                        k8, v8t, vitfp8_vt_stride(total_tokens), stream) == cudaSuccess
               ? VITFP8_OK
               : VITFP8_ERR_CUDA;
}

size_t vitfp8_attn_workspace_size(int32_t num_seqs) {
    if (num_seqs < 0) return 0;
    return ws_bytes(num_seqs);
}

static_assert(VITFP8_ATTN_AUTO == kAttnAuto && VITFP8_ATTN_UNIT == kAttnUnit &&
                  VITFP8_ATTN_PERSISTENT == kAttnPersistent && VITFP8_ATTN_TWO_TILE == kAttnTwoTile &&
                  VITFP8_ATTN_TWO_TILE_PERSISTENT == kAttnTwoTilePersistent,
              "kernel numbers of the header and the launcher agree");

vitfp8_status vitfp8_attn_varlen_kernel(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                                        const vitfp8_scale_state* d_state, const int32_t* d_cu_seqlens,
                                        int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                        int32_t H, int32_t D, int32_t D_pad, float sm_scale,
                                        vitfp8_bf16* out, void* d_workspace, size_t workspace_bytes,
                                        int32_t kernel, cudaStream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H <= 0) return VITFP8_ERR_INVALID_ARG;
    if (D < 8 || (D & 7) || D_pad < D || (D_pad & 15)) return VITFP8_ERR_INVALID_ARG;
    if (kernel < VITFP8_ATTN_AUTO || kernel > VITFP8_ATTN_TWO_TILE_PERSISTENT) return VITFP8_ERR_INVALID_ARG;
    if (D > VITFP8_MAX_HEAD_DIM || D_pad > VITFP8_MAX_HEAD_DIM) return VITFP8_ERR_UNSUPPORTED;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f)) return VITFP8_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_tokens == 0) return VITFP8_OK;
    if (!q8 || !k8 || !v8t || !d_state || !d_cu_seqlens || !out) return VITFP8_ERR_INVALID_ARG;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(out) ||
        !aligned4(d_state) || !aligned4(d_cu_seqlens))
        return VITFP8_ERR_INVALID_ARG;
    if (!d_workspace || !aligned16(d_workspace) || workspace_bytes < ws_bytes(num_seqs))
        return VITFP8_ERR_WORKSPACE;
    return launch_attn_fp8(q8, k8, v8t, d_state, d_cu_seqlens, num_seqs, max_seqlen, total_tokens, H, D, D_pad,
                           vitfp8_vt_stride(total_tokens), sm_scale,
                           reinterpret_cast<uint16_t*>(out), d_workspace, kernel, stream);
}

vitfp8_status vitfp8_attn_varlen(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                                 const vitfp8_scale_state* d_state, const int32_t* d_cu_seqlens,
                                 int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                 int32_t H, int32_t D, int32_t D_pad, float sm_scale,
                                 vitfp8_bf16* out, void* d_workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    return vitfp8_attn_varlen_kernel(q8, k8, v8t, d_state, d_cu_seqlens, num_seqs, max_seqlen, total_tokens,
                                     H, D, D_pad, sm_scale, out, d_workspace, workspace_bytes,
                                     VITFP8_ATTN_AUTO, stream);
}

int32_t vitfp8_attn_kernel_for(int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens, int32_t H,
                               int32_t num_sms) {
    return attn_fp8_kernel_for(num_seqs, max_seqlen, total_tokens, H, num_sms);
}

vitfp8_status vitfp8_attn_varlen_bf16(const vitfp8_bf16* q, const vitfp8_bf16* k,
                                      const vitfp8_bf16* v, const int32_t* d_cu_seqlens,
                                      int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                      int32_t H, int32_t D, float sm_scale, vitfp8_bf16* out,
                                      void* d_workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
    if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || H <= 0) return VITFP8_ERR_INVALID_ARG;
    if (D < 8 || (D & 7)) return VITFP8_ERR_INVALID_ARG;
    if (D > VITFP8_MAX_HEAD_DIM) return VITFP8_ERR_UNSUPPORTED;
    if (!std::isfinite(sm_scale) || !(sm_scale > 0.0f)) return VITFP8_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_tokens == 0) return VITFP8_OK;
    if (!q || !k || !v || !d_cu_seqlens || !out) return VITFP8_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned4(d_cu_seqlens))
        return VITFP8_ERR_INVALID_ARG;
    if (!d_workspace || !aligned16(d_workspace) || workspace_bytes < ws_bytes(num_seqs))
        return VITFP8_ERR_WORKSPACE;
    return launch_attn_bf16(reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k),
                            reinterpret_cast<const uint16_t*>(v), d_cu_seqlens, num_seqs, max_seqlen,
                            total_tokens, H, D, sm_scale, reinterpret_cast<uint16_t*>(out),
                            d_workspace, stream);
}

vitfp8_status vitfp8_get_device_error(const vitfp8_scale_state* d_state, int32_t* h_out,
                                      cudaStream_t stream) {
    if (!d_state || !h_out) return VITFP8_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return VITFP8_ERR_CUDA;
    if (cudaMemcpy(h_out, &d_state->dev_error, sizeof(int32_t), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return VITFP8_ERR_CUDA;
    return VITFP8_OK;
}

vitfp8_status vitfp8_selftest_bounded_wait(void* d_workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
    if (!d_workspace || workspace_bytes < sizeof(WsHeader) || !aligned4(d_workspace))
        return VITFP8_ERR_INVALID_ARG;
    return launch_selftest_wait(d_workspace, stream) == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

vitfp8_status vitfp8_selftest_bounds_check(void* d_workspace, size_t workspace_bytes,
                                           cudaStream_t stream) {
    if (!d_workspace || workspace_bytes < sizeof(WsHeader) || !aligned4(d_workspace))
        return VITFP8_ERR_INVALID_ARG;
    return launch_selftest_bounds(d_workspace, stream) == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

int32_t vitfp8_checked_build(void) { return VF_CHECKED_BUILD; }

vitfp8_status vitfp8_get_workspace_error(const void* d_workspace, int32_t* h_out,
                                         cudaStream_t stream) {
    if (!d_workspace || !h_out) return VITFP8_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return VITFP8_ERR_CUDA;
    const WsHeader* hdr = static_cast<const WsHeader*>(d_workspace);
    if (cudaMemcpy(h_out, &hdr->error, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return VITFP8_ERR_CUDA;
    return VITFP8_OK;
}

}  // extern "C"
