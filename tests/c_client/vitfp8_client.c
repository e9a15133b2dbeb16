/*
 * A plain C client of the library, for the tests: it uses only the C ABI of
 * vitfp8.h and the CUDA runtime (no Python, no torch types), the way an
 * inference runtime would.
 *
 *   vitfp8_client IN OUT
 *
 * IN:  int32 T, H, D, nseq, forwards; int32 cu_seqlens[nseq + 1]; then for
 *      each forward bf16 q, k, v, each [T][H][D] (raw 16-bit patterns).
 * OUT: the vitfp8_scale_state after the last forward (raw bytes), the bf16
 *      attention output [T][H][D] of the last forward, then the three
 *      scale-file values (float32, q k v) vitfp8_calibrated_scales gives for
 *      that state with margin 1.5.
 *
 * Each forward runs dynamic scaling, quantization with un-padding and FP8
 * attention on one stream.  Every status is checked; the exit code is 0 only
 * if every call and both device error words report success.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "vitfp8.h"

#define CK_CUDA(x)                                                        \
    do {                                                                  \
        cudaError_t e_ = (x);                                             \
        if (e_ != cudaSuccess) {                                          \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));      \
            return 2;                                                     \
        }                                                                 \
    } while (0)
#define CK_VF(x)                                                          \
    do {                                                                  \
        vitfp8_status s_ = (x);                                           \
        if (s_ != VITFP8_OK) {                                            \
            fprintf(stderr, "%s: %s\n", #x, vitfp8_status_string(s_));    \
            return 3;                                                     \
        }                                                                 \
    } while (0)

static int read_all(FILE* f, void* dst, size_t n) { return fread(dst, 1, n, f) == n ? 0 : -1; }

int main(int argc, char** argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s IN OUT\n", argv[0]);
        return 1;
    }
    FILE* in = fopen(argv[1], "rb");
    if (!in) return 1;
    int32_t hdr[5];
    if (read_all(in, hdr, sizeof(hdr))) return 1;
    const int32_t T = hdr[0], H = hdr[1], D = hdr[2], nseq = hdr[3], forwards = hdr[4];
    const int32_t Dp = (D + 15) / 16 * 16;
    const size_t n_elem = (size_t)T * H * D;
    int32_t* h_cu = (int32_t*)malloc(sizeof(int32_t) * (nseq + 1));
    vitfp8_bf16* h_src = (vitfp8_bf16*)malloc(3 * n_elem * sizeof(vitfp8_bf16));
    vitfp8_bf16* h_out = (vitfp8_bf16*)malloc(n_elem * sizeof(vitfp8_bf16));
    if (!h_cu || !h_src || !h_out || read_all(in, h_cu, sizeof(int32_t) * (nseq + 1))) return 1;

    const int64_t Tv = vitfp8_vt_stride(T);
    const size_t ws_bytes = vitfp8_attn_workspace_size(nseq);
    vitfp8_scale_state* d_state;
    int32_t* d_cu;
    vitfp8_bf16 *d_src, *d_out;
    uint8_t *d_q8, *d_k8, *d_v8t;
    void* d_ws;
    CK_CUDA(cudaMalloc((void**)&d_state, sizeof(vitfp8_scale_state)));
    CK_CUDA(cudaMalloc((void**)&d_cu, sizeof(int32_t) * (nseq + 1)));
    CK_CUDA(cudaMalloc((void**)&d_src, 3 * n_elem * sizeof(vitfp8_bf16) + 16));
    CK_CUDA(cudaMalloc((void**)&d_out, n_elem * sizeof(vitfp8_bf16) + 16));
    CK_CUDA(cudaMalloc((void**)&d_q8, (size_t)T * H * Dp + 16));
    CK_CUDA(cudaMalloc((void**)&d_k8, (size_t)T * H * Dp + 16));
    CK_CUDA(cudaMalloc((void**)&d_v8t, (size_t)H * Dp * Tv + 16));
    CK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    cudaStream_t s;
    CK_CUDA(cudaStreamCreate(&s));
    CK_CUDA(cudaMemcpyAsync(d_cu, h_cu, sizeof(int32_t) * (nseq + 1), cudaMemcpyHostToDevice, s));
    CK_VF(vitfp8_scale_state_init(d_state, s));

    const vitfp8_src_layout lay = {0, 0, 0, (int64_t)H * D, D};   /* packed [T][H][D] */
    const vitfp8_bf16* d_q = d_src;
    const vitfp8_bf16* d_k = d_src + n_elem;
    const vitfp8_bf16* d_v = d_src + 2 * n_elem;
    const float sm_scale = (float)(1.0 / sqrt((double)D));
    int32_t max_seqlen = 0;
    for (int32_t b = 0; b < nseq; ++b)
        if (h_cu[b + 1] - h_cu[b] > max_seqlen) max_seqlen = h_cu[b + 1] - h_cu[b];
    for (int32_t f = 0; f < forwards; ++f) {
        if (read_all(in, h_src, 3 * n_elem * sizeof(vitfp8_bf16))) return 1;
        CK_CUDA(cudaMemcpyAsync(d_src, h_src, 3 * n_elem * sizeof(vitfp8_bf16), cudaMemcpyHostToDevice, s));
        CK_VF(vitfp8_amax_update(d_state, d_q, d_k, d_v, &lay, d_cu, nseq, T, H, D, s));
        CK_VF(vitfp8_quantize_unpad(d_state, d_q, d_k, d_v, &lay, d_cu, nseq, T, H, D, Dp, d_q8, d_k8,
                                    d_v8t, s));
        CK_VF(vitfp8_attn_varlen(d_q8, d_k8, d_v8t, d_state, d_cu, nseq, max_seqlen, T, H, D, Dp,
                                 sm_scale, d_out, d_ws, ws_bytes, s));
        /* the host buffer is refilled next iteration: finish this forward's copy first */
        CK_CUDA(cudaStreamSynchronize(s));
    }
    fclose(in);

    /* The last forward's codes through each named kernel (unit, persistent,
     * two-tile, persistent two-tile), and the kernel the host rule picks. */
    vitfp8_bf16* h_kout = (vitfp8_bf16*)malloc(4 * n_elem * sizeof(vitfp8_bf16));
    vitfp8_bf16* d_kout;
    if (!h_kout) return 1;
    CK_CUDA(cudaMalloc((void**)&d_kout, 4 * n_elem * sizeof(vitfp8_bf16)));
    for (int32_t kern = VITFP8_ATTN_UNIT; kern <= VITFP8_ATTN_TWO_TILE_PERSISTENT; ++kern)
        CK_VF(vitfp8_attn_varlen_kernel(d_q8, d_k8, d_v8t, d_state, d_cu, nseq, max_seqlen, T, H, D, Dp,
                                        sm_scale, d_kout + (size_t)(kern - 1) * n_elem, d_ws, ws_bytes,
                                        kern, s));
    if (vitfp8_attn_varlen_kernel(d_q8, d_k8, d_v8t, d_state, d_cu, nseq, max_seqlen, T, H, D, Dp, sm_scale,
                                  d_kout, d_ws, ws_bytes, 99, s) != VITFP8_ERR_INVALID_ARG)
        return 5;
    int32_t picked = vitfp8_attn_kernel_for(nseq, max_seqlen, T, H, 152);
    if (picked < VITFP8_ATTN_UNIT || picked > VITFP8_ATTN_TWO_TILE_PERSISTENT) return 6;
    CK_CUDA(cudaMemcpyAsync(h_kout, d_kout, 4 * n_elem * sizeof(vitfp8_bf16), cudaMemcpyDeviceToHost, s));

    /* Calibrate once from C: the scale-file values of this state (margin 1.5). */
    float* d_saved;
    float h_saved[3];
    CK_CUDA(cudaMalloc((void**)&d_saved, 3 * sizeof(float)));
    CK_VF(vitfp8_calibrated_scales(d_state, 1.5f, d_saved, NULL, s));
    CK_CUDA(cudaMemcpyAsync(h_saved, d_saved, sizeof(h_saved), cudaMemcpyDeviceToHost, s));

    int32_t dev_err = -1, ws_err = -1;
    CK_VF(vitfp8_get_device_error(d_state, &dev_err, s));
    CK_VF(vitfp8_get_workspace_error(d_ws, &ws_err, s));
    vitfp8_scale_state h_state;
    CK_CUDA(cudaMemcpy(&h_state, d_state, sizeof(h_state), cudaMemcpyDeviceToHost));
    CK_CUDA(cudaMemcpy(h_out, d_out, n_elem * sizeof(vitfp8_bf16), cudaMemcpyDeviceToHost));
    FILE* out = fopen(argv[2], "wb");
    if (!out) return 1;
    if (fwrite(&h_state, sizeof(h_state), 1, out) != 1 ||
        fwrite(h_out, sizeof(vitfp8_bf16), n_elem, out) != n_elem ||
        fwrite(h_saved, sizeof(float), 3, out) != 3 ||
        fwrite(h_kout, sizeof(vitfp8_bf16), 4 * n_elem, out) != 4 * n_elem)
        return 1;
    fclose(out);
    printf("vitfp8 %d: device error %d, workspace error %d\n", vitfp8_version(), dev_err, ws_err);
    return (dev_err == 0 && ws_err == 0) ? 0 : 4;
}
