// Dynamic amax + 16-entry ring update, and quantize + un-pad of Q, K, V.
//
// "FP8 ViT Encoder Attention", Usage: a 16-entry circular buffer of observed
// Q/K/V amax values drives per-forward scale updates; intro and note: Q/K/V are
// quantized on the fly to FP8 before the attention call, with "quantization
// kernel launches + un-padding".  Here both steps cover q, k and v in ONE
// launch each (the pages cite three quantization launches plus un-padding).
//
// Both kernels are HBM-bound streams: 16-byte vector loads of 8 bf16 values,
// coalesced along the head dim, tiles of 64 tokens x one head per block.
// Every computed index passes VF_IN (checked.cuh): a no-op in the normal
// build, a bounds check into the device error word in the checked build.
#include <cuda_runtime.h>

#include "checked.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

constexpr int QT_TOK = 64;       // tokens per block tile
constexpr int QT_THREADS = 256;  // threads per block
constexpr int MAX_DP = 256;      // largest padded head dim the quant kernel takes

// ---------------------------------------------------------------- helpers

// Source row of packed token t (padded batch: b * s_max + i; packed: t), or -1
// if cu_seqlens puts t outside its segment's padded rows.
__device__ __forceinline__ int64_t src_row_of(const SrcDev& L, const int32_t* cu, int nseq, int t,
                                              int32_t* err) {
    if (!L.padded) return t;
    int lo = 0, hi = nseq - 1;  // largest b with cu[b] <= t
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (!VF_IN(mid, 1, nseq + 1, err)) return -1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    if (!VF_IN(lo, 1, nseq + 1, err)) return -1;
    int64_t i = int64_t(t) - __ldg(cu + lo);
    if (i < 0 || i >= L.s_max) {
        record_error(err, VITFP8_ERR_BAD_SEQLENS);
        return -1;
    }
    return int64_t(lo) * L.s_max + i;
}

// Not volatile: the inputs are read-only for the kernel's duration, so the
// compiler may hoist several of these loads ahead of the arithmetic that uses
// them (they are then in flight together).
__device__ __forceinline__ uint4 ld_stream16(const uint16_t* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Running max of |x| over two bf16 lanes, as 16-bit magnitude patterns.  For
// non-NaN values the magnitude bits order like the magnitudes; NaN patterns
// (above 0x7F80) are dropped (fmax semantics), +inf (0x7F80) is kept.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t m, uint32_t w) {
    uint32_t a = w & 0x7FFF7FFFu;
    uint32_t nan = __vcmpgtu2(a, 0x7F807F80u);
    return __vmaxu2(m, a & ~nan);
}

// 4 bf16 (two words) -> 4 E4M3 codes of float32(x) * inv.
__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, float inv) {
    float y0 = __fmul_rn(__uint_as_float(w0 << 16), inv);
    float y1 = __fmul_rn(__uint_as_float(w0 & 0xFFFF0000u), inv);
    float y2 = __fmul_rn(__uint_as_float(w1 << 16), inv);
    float y3 = __fmul_rn(__uint_as_float(w1 & 0xFFFF0000u), inv);
    return cvt_e4m3x2(y0, y1) | (cvt_e4m3x2(y2, y3) << 16);
}

__device__ __forceinline__ void scale_from_amax(float A, float& sc, float& inv) {
    if (A == 0.0f) {
        sc = 1.0f;
        inv = 1.0f;
    } else {
        sc = __fdiv_rn(A, VITFP8_E4M3_MAX);
        inv = __fdiv_rn(VITFP8_E4M3_MAX, A);
    }
}

// ---------------------------------------------------------------- state

__global__ void state_init_kernel(vitfp8_scale_state* st) {
    for (int t = 0; t < 3; ++t) {
        for (int i = 0; i < VITFP8_RING; ++i) st->hist[t][i] = 0.0f;
        st->amax_ref[t] = 0.0f;
        st->scale[t] = 1.0f;
        st->inv_scale[t] = 1.0f;
        st->amax_cur[t] = 0.0f;
        st->amax_bits[t] = 0u;
    }
    st->pos = 0;
    st->count = 0;
    st->mode = 0;
    st->dev_error = 0;
    st->blocks_done = 0u;
}

__global__ void set_static_kernel(vitfp8_scale_state* st, float q, float k, float v) {
    const float a[3] = {q, k, v};
    st->mode = 1;
    for (int t = 0; t < 3; ++t) {
        st->amax_ref[t] = a[t];
        scale_from_amax(a[t], st->scale[t], st->inv_scale[t]);
    }
}

// ---------------------------------------------------------------- amax

// Reference and scales from the ring maximum.  One thread.
__device__ void scale_from_ring(vitfp8_scale_state* st) {
    for (int t = 0; t < 3; ++t) {
        float A = 0.0f;
        for (int i = 0; i < VITFP8_RING; ++i) A = fmaxf(A, st->hist[t][i]);
        st->amax_ref[t] = A;
        scale_from_amax(A, st->scale[t], st->inv_scale[t]);
    }
}

// One dynamic forward's ring update with (a_q, a_k, a_v).  Mode 0: push,
// then scale from the ring including the push.  Mode 2 (delayed scaling):
// scale from the ring the earlier forwards left, then push.  One thread.
__device__ void ring_push_scale(vitfp8_scale_state* st, const float (&a)[3]) {
    const bool delayed = st->mode == 2;
    if (delayed) scale_from_ring(st);
    const int pos = st->pos;
    if (!VF_IN(pos, 1, VITFP8_RING, &st->dev_error)) return;
    for (int t = 0; t < 3; ++t) {
        st->amax_cur[t] = a[t];
        st->hist[t][pos] = a[t];
    }
    st->pos = (pos + 1) % VITFP8_RING;
    st->count = min(st->count + 1, VITFP8_RING);
    if (!delayed) scale_from_ring(st);
}

__global__ void set_ring_order_kernel(vitfp8_scale_state* st, int delayed) {
    if (st->mode != 1) st->mode = delayed ? 2 : 0;
}

// Block maximum of m (two bf16 magnitudes per 32-bit lane), one atomicMax into
// the tensor's reduction word, and the launch's last block (atomic counter;
// no grid barrier, no spin) either pushes the forward's amax into the ring or,
// with `out`, writes (a_q, a_k, a_v, 1) there.
__device__ __forceinline__ void amax_block_finish(vitfp8_scale_state* st, int z, uint32_t m,
                                                  float* out, uint32_t* wmax) {
    m = max(m & 0xFFFFu, m >> 16);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0 && VF_IN(threadIdx.x >> 5, 1, QT_THREADS / 32, &st->dev_error))
        wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x != 0) return;

    uint32_t bm = 0;
#pragma unroll
    for (int w = 0; w < QT_THREADS / 32; ++w) bm = max(bm, wmax[w]);
    if (bm) atomicMax(&st->amax_bits[z], bm);
    __threadfence();
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    const unsigned prev = atomicAdd(&st->blocks_done, 1u);
    if (prev != total - 1) return;

    // Last block: every other block's atomicMax is visible.
    __threadfence();
    float a[3];
    for (int t = 0; t < 3; ++t) {
        const uint32_t bits = atomicExch(&st->amax_bits[t], 0u);
        a[t] = __uint_as_float(bits << 16);
    }
    if (out) {
        for (int t = 0; t < 3; ++t) {
            st->amax_cur[t] = a[t];
            out[t] = a[t];
        }
        out[3] = 1.0f;
    } else {
        ring_push_scale(st, a);
    }
    st->blocks_done = 0u;
}

// `out` null: the last block pushes the forward's amax into the ring.
// `out` non-null (data-parallel step 1): the last block writes
// (a_q, a_k, a_v, 1) there instead and leaves the ring alone; in static mode
// block 0 writes zeros (nothing to reduce, nothing to push).
__global__ void __launch_bounds__(QT_THREADS)
amax_kernel(vitfp8_scale_state* st, const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
            const uint16_t* __restrict__ v, SrcDev L, const int32_t* __restrict__ cu, int nseq,
            int T, int H, int D, float* __restrict__ out) {
    if (st->mode == 1) {  // static mode: nothing to track
        if (out && threadIdx.x < 4 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
            VF_IN(threadIdx.x, 1, 4, &st->dev_error))
            out[threadIdx.x] = 0.0f;
        return;
    }
    const int z = blockIdx.z;
    const uint16_t* src = z == 0 ? q : (z == 1 ? k : v);
    const int t0 = blockIdx.x * QT_TOK;
    const int h = blockIdx.y;
    __shared__ int64_t rows[QT_TOK];
    __shared__ uint32_t wmax[QT_THREADS / 32];
    if (threadIdx.x < QT_TOK) {
        const int t = t0 + threadIdx.x;
        rows[threadIdx.x] = t < T ? src_row_of(L, cu, nseq, t, &st->dev_error) : -1;
    }
    __syncthreads();

    const int VD = D >> 3;
    const int nvec = QT_TOK * VD;
    const int64_t hoff = int64_t(h) * L.hs;
    uint32_t m = 0;
    for (int base = threadIdx.x; base < nvec; base += 4 * QT_THREADS) {
        uint4 w[4];
        bool ok[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * QT_THREADS;
            const int tt = i / VD;
            const int c = i - tt * VD;
            ok[u] = i < nvec && rows[tt < QT_TOK ? tt : 0] >= 0;
            if (ok[u]) ok[u] = VF_IN(tt, 1, QT_TOK, &st->dev_error) &&
                               VF_IN(rows[tt] * L.ts + hoff + c * 8, 8, L.extent, &st->dev_error);
            w[u] = ok[u] ? ld_stream16(src + rows[tt] * L.ts + hoff + c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            m = absmax_bf16x2(m, w[u].x);
            m = absmax_bf16x2(m, w[u].y);
            m = absmax_bf16x2(m, w[u].z);
            m = absmax_bf16x2(m, w[u].w);
        }
    }
    amax_block_finish(st, z, m, out, wmax);
}

// Same reduction when each token's heads are contiguous (head stride == D,
// e.g. packed [T, H, D] or a fused QKV view): the amax is one value per
// tensor, so a block reads whole token rows of H * D elements (long
// coalesced runs) instead of one head's D-element slice per token.  Grid
// (blocks, 1, 3); each block walks 16-token tiles, each warp two tokens of a
// tile, 32 lanes x 16 bytes per step.
constexpr int AR_TOK = 16;
static_assert(AR_TOK == 2 * (QT_THREADS / 32), "two tokens of a tile per warp");
// At least 4 resident blocks per SM: up to 64 registers, so that a warp's 16
// loads of a tile are in flight together (at 8 blocks the compiler keeps to
// 32 registers and a few loads at a time).
__global__ void __launch_bounds__(QT_THREADS, 4)
amax_rows_kernel(vitfp8_scale_state* st, const uint16_t* __restrict__ q,
                 const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, SrcDev L,
                 const int32_t* __restrict__ cu, int nseq, int T, int H, int D,
                 float* __restrict__ out) {
    if (st->mode == 1) {
        if (out && threadIdx.x < 4 && blockIdx.x == 0 && blockIdx.z == 0 &&
            VF_IN(threadIdx.x, 1, 4, &st->dev_error))
            out[threadIdx.x] = 0.0f;
        return;
    }
    const int z = blockIdx.z;
    const uint16_t* src = z == 0 ? q : (z == 1 ? k : v);
    __shared__ int64_t rows[AR_TOK];
    __shared__ uint32_t wmax[QT_THREADS / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RV = H * (D >> 3);   // 16-byte vectors per token row
    const int ntiles = (T + AR_TOK - 1) / AR_TOK;
    uint32_t m = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        __syncthreads();   // the previous tile's rows[] are no longer read
        if (threadIdx.x < AR_TOK) {
            const int t = tile * AR_TOK + threadIdx.x;
            rows[threadIdx.x] = t < T ? src_row_of(L, cu, nseq, t, &st->dev_error) : -1;
        }
        __syncthreads();
        // Warp w reads tokens w and w + 8 of the tile: both rows' 16-byte
        // vectors, 8 per lane and row, are in flight before any is reduced.
        const int64_t rowA = rows[warp], rowB = rows[warp + QT_THREADS / 32];
        for (int j0 = 0; j0 < RV; j0 += 8 * 32) {
            uint4 w[16];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + lane + 32 * u;
                w[u] = (rowA >= 0 && j < RV &&
                        VF_IN(rowA * L.ts + int64_t(j) * 8, 8, L.extent, &st->dev_error))
                           ? ld_stream16(src + rowA * L.ts + int64_t(j) * 8)
                           : make_uint4(0, 0, 0, 0);
                w[8 + u] = (rowB >= 0 && j < RV &&
                            VF_IN(rowB * L.ts + int64_t(j) * 8, 8, L.extent, &st->dev_error))
                               ? ld_stream16(src + rowB * L.ts + int64_t(j) * 8)
                               : make_uint4(0, 0, 0, 0);
            }
            // Every load above is issued before the reduction starts.
            asm volatile("" : "+r"(w[0].x), "+r"(w[1].x), "+r"(w[2].x), "+r"(w[3].x), "+r"(w[4].x), "+r"(w[5].x),
                              "+r"(w[6].x), "+r"(w[7].x), "+r"(w[8].x), "+r"(w[9].x), "+r"(w[10].x), "+r"(w[11].x),
                              "+r"(w[12].x), "+r"(w[13].x), "+r"(w[14].x), "+r"(w[15].x));
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                m = absmax_bf16x2(m, w[u].x);
                m = absmax_bf16x2(m, w[u].y);
                m = absmax_bf16x2(m, w[u].z);
                m = absmax_bf16x2(m, w[u].w);
            }
        }
    }
    amax_block_finish(st, z, m, out, wmax);
}

// Data-parallel step 3: push reduced values (a_q, a_k, a_v, any) if any > 0.
__global__ void ring_push_kernel(vitfp8_scale_state* st, const float* __restrict__ vals) {
    if (st->mode == 1 || !(vals[3] > 0.0f)) return;
    const float a[3] = {vals[0], vals[1], vals[2]};
    ring_push_scale(st, a);
}

// ---------------------------------------------------------------- quantize

__global__ void __launch_bounds__(QT_THREADS)
quant_kernel(const vitfp8_scale_state* __restrict__ st, const uint16_t* __restrict__ q,
             const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, SrcDev L,
             const int32_t* __restrict__ cu, int nseq, int T, int H, int D, int Dp,
             uint8_t* __restrict__ q8, uint8_t* __restrict__ k8, uint8_t* __restrict__ v8t,
             int64_t Tv, int32_t* err, int rows_tok) {
    const int z = blockIdx.z;
    const uint16_t* src = z == 0 ? q : (z == 1 ? k : v);
    if (z < 2 && rows_tok > 0) {
        // Q and K with contiguous heads and no d padding (head stride == D ==
        // D_pad): source and code rows are flat runs of H * D elements, so
        // this block converts whole token rows -- `rows_tok` tokens from the
        // block's flat index -- instead of one head's slice.  The grid is
        // the one V's per-head transpose needs; rows_tok = ceil(64 / H)
        // makes the row blocks cover all T tokens within it.
        const int64_t flat = int64_t(blockIdx.y) * gridDim.x + blockIdx.x;
        const int64_t r0 = flat * rows_tok;
        if (r0 >= T) return;
        const int RV = H * (D >> 3);
        const float inv = st->inv_scale[z];
        uint8_t* dst0 = z == 0 ? q8 : k8;
        for (int tt = 0; tt < rows_tok; tt += 4) {
            int64_t srow[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t t = r0 + tt + u;
                srow[u] = (tt + u < rows_tok && t < T) ? src_row_of(L, cu, nseq, int(t), err) : -1;
            }
            for (int j = threadIdx.x; j < RV; j += QT_THREADS) {
                uint4 w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w[u] = (srow[u] >= 0 && VF_IN(srow[u] * L.ts + int64_t(j) * 8, 8, L.extent, err))
                               ? ld_stream16(src + srow[u] * L.ts + int64_t(j) * 8)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t t = r0 + tt + u;
                    if (tt + u >= rows_tok || t >= T) continue;
                    uint2 o = make_uint2(0u, 0u);
                    if (srow[u] >= 0) {
                        o.x = quant4(w[u].x, w[u].y, inv);
                        o.y = quant4(w[u].z, w[u].w, inv);
                    }
                    if (VF_IN(t * (int64_t(H) * Dp) + int64_t(j) * 8, 8, int64_t(T) * H * Dp, err))
                        *reinterpret_cast<uint2*>(dst0 + t * (int64_t(H) * Dp) + int64_t(j) * 8) = o;
                }
            }
        }
        return;
    }
    const int t0 = blockIdx.x * QT_TOK;
    const int h = blockIdx.y;
    __shared__ int64_t rows[QT_TOK];
    // V transpose tile: QT_TOK token rows of Dp code bytes, padded by one word
    // per row to spread banks.
    __shared__ uint32_t tile[QT_TOK * (MAX_DP / 4 + 1)];
    if (threadIdx.x < QT_TOK) {
        const int t = t0 + threadIdx.x;
        rows[threadIdx.x] = t < T ? src_row_of(L, cu, nseq, t, err) : -1;
    }
    __syncthreads();

    const float inv = st->inv_scale[z];
    const int VD = D >> 3;   // source vectors per row
    const int VP = Dp >> 3;  // output 8-byte groups per row
    const int nvec = QT_TOK * VP;
    const int64_t hoff = int64_t(h) * L.hs;
    const int SW = Dp / 4 + 1;

    for (int base = threadIdx.x; base < nvec; base += 4 * QT_THREADS) {
        uint4 w[4];
        bool ld[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * QT_THREADS;
            const int tt = i / VP;
            const int c = i - tt * VP;
            ld[u] = i < nvec && c < VD && rows[tt < QT_TOK ? tt : 0] >= 0;
            if (ld[u]) ld[u] = VF_IN(tt, 1, QT_TOK, err) && VF_IN(rows[tt] * L.ts + hoff + c * 8, 8, L.extent, err);
            w[u] = ld[u] ? ld_stream16(src + rows[tt] * L.ts + hoff + c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = base + u * QT_THREADS;
            if (i >= nvec) continue;
            const int tt = i / VP;
            const int c = i - tt * VP;
            uint2 o = make_uint2(0u, 0u);
            if (ld[u]) {
                o.x = quant4(w[u].x, w[u].y, inv);
                o.y = quant4(w[u].z, w[u].w, inv);
            }
            if (z < 2) {
                const int t = t0 + tt;
                if (t < T && VF_IN((int64_t(t) * H + h) * Dp + c * 8, 8, int64_t(T) * H * Dp, err)) {
                    uint8_t* dst = (z == 0 ? q8 : k8) + (int64_t(t) * H + h) * Dp + c * 8;
                    *reinterpret_cast<uint2*>(dst) = o;
                }
            } else if (VF_IN(tt * SW + 2 * c, 2, QT_TOK * (MAX_DP / 4 + 1), err)) {
                tile[tt * SW + 2 * c] = o.x;
                tile[tt * SW + 2 * c + 1] = o.y;
            }
        }
    }
    if (z < 2) return;

    // V: write [h][d][t] rows of 4 tokens x 4 d at a time (4x4 byte transpose).
    __syncthreads();
    const int nq = (Dp / 4) * (QT_TOK / 4);
    for (int i = threadIdx.x; i < nq; i += QT_THREADS) {
        const int tq = i % (QT_TOK / 4);
        const int dq = i / (QT_TOK / 4);
        const int tt = tq * 4;
        const int64_t t = int64_t(t0) + tt;
        if (t >= Tv) continue;
        if (!VF_IN((tt + 3) * SW + dq, 1, QT_TOK * (MAX_DP / 4 + 1), err)) continue;
        const uint32_t w0 = tile[(tt + 0) * SW + dq];
        const uint32_t w1 = tile[(tt + 1) * SW + dq];
        const uint32_t w2 = tile[(tt + 2) * SW + dq];
        const uint32_t w3 = tile[(tt + 3) * SW + dq];
        const uint32_t a0 = __byte_perm(w0, w1, 0x5140);
        const uint32_t a1 = __byte_perm(w2, w3, 0x5140);
        const uint32_t a2 = __byte_perm(w0, w1, 0x7362);
        const uint32_t a3 = __byte_perm(w2, w3, 0x7362);
        const uint32_t o[4] = {__byte_perm(a0, a1, 0x5410), __byte_perm(a0, a1, 0x7632),
                               __byte_perm(a2, a3, 0x5410), __byte_perm(a2, a3, 0x7632)};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (VF_IN((int64_t(h) * Dp + dq * 4 + j) * Tv + t, 4, int64_t(H) * Dp * Tv, err))
                *reinterpret_cast<uint32_t*>(v8t + (int64_t(h) * Dp + dq * 4 + j) * Tv + t) = o[j];
    }
}

// ---------------------------------------------------------------- calibrate once

// Calibrate-once step on the device: for each tensor the ring maximum A of
// the calibrated dynamic state, the saved value float32(A) * float32(margin)
// written to `out` (if given), and the static state `dst` (if given) set from
// those values exactly as vitfp8_set_static_scales would.  A tensor whose ring
// holds no amax (A == 0) makes no valid static scale: the dynamic state's
// error word records VITFP8_ERR_INVALID_ARG and `dst` is left as it is.  One
// thread.
__global__ void calibrated_scales_kernel(vitfp8_scale_state* dyn, float margin, float* out,
                                         vitfp8_scale_state* dst) {
    float saved[3];
    bool ok = true;
    for (int t = 0; t < 3; ++t) {
        float A = 0.0f;
        for (int i = 0; i < VITFP8_RING; ++i) A = fmaxf(A, dyn->hist[t][i]);
        saved[t] = __fmul_rn(A, margin);
        ok = ok && saved[t] > 0.0f && saved[t] <= 3.4028234e38f;
        if (out) out[t] = saved[t];
    }
    if (!ok) {
        record_error(&dyn->dev_error, VITFP8_ERR_INVALID_ARG);
        return;
    }
    if (dst) {
        dst->mode = 1;
        for (int t = 0; t < 3; ++t) {
            dst->amax_ref[t] = saved[t];
            scale_from_amax(saved[t], dst->scale[t], dst->inv_scale[t]);
        }
    }
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_state_init(vitfp8_scale_state* st, cudaStream_t s) {
    state_init_kernel<<<1, 1, 0, s>>>(st);
    return cudaGetLastError();
}

cudaError_t launch_set_static(vitfp8_scale_state* st, float q, float k, float v, cudaStream_t s) {
    set_static_kernel<<<1, 1, 0, s>>>(st, q, k, v);
    return cudaGetLastError();
}

cudaError_t launch_amax(vitfp8_scale_state* st, const uint16_t* q, const uint16_t* k,
                        const uint16_t* v, SrcDev L, const int32_t* cu, int nseq, int T, int H,
                        int D, float* out, cudaStream_t s) {
    if (L.hs == D) {
        // one 16-token tile per block up to 1024 blocks per tensor (about 4
        // resident blocks of 256 threads per SM), then tiles walked by stride
        const int ntiles = (T + AR_TOK - 1) / AR_TOK;
        dim3 grid(ntiles < 1024 ? ntiles : 1024, 1, 3);
        amax_rows_kernel<<<grid, QT_THREADS, 0, s>>>(st, q, k, v, L, cu, nseq, T, H, D, out);
    } else {
        dim3 grid((T + QT_TOK - 1) / QT_TOK, H, 3);
        amax_kernel<<<grid, QT_THREADS, 0, s>>>(st, q, k, v, L, cu, nseq, T, H, D, out);
    }
    return cudaGetLastError();
}

cudaError_t launch_set_ring_order(vitfp8_scale_state* st, int delayed, cudaStream_t s) {
    set_ring_order_kernel<<<1, 1, 0, s>>>(st, delayed);
    return cudaGetLastError();
}

cudaError_t launch_calibrated_scales(const vitfp8_scale_state* dyn, float margin, float* out,
                                     vitfp8_scale_state* dst, cudaStream_t s) {
    calibrated_scales_kernel<<<1, 1, 0, s>>>(const_cast<vitfp8_scale_state*>(dyn), margin, out, dst);
    return cudaGetLastError();
}

cudaError_t launch_ring_push(vitfp8_scale_state* st, const float* vals, cudaStream_t s) {
    ring_push_kernel<<<1, 1, 0, s>>>(st, vals);
    return cudaGetLastError();
}

cudaError_t launch_quant(const vitfp8_scale_state* st, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, SrcDev L, const int32_t* cu, int nseq, int T, int H,
                         int D, int Dp, uint8_t* q8, uint8_t* k8, uint8_t* v8t, int64_t Tv,
                         cudaStream_t s) {
    dim3 grid((T + QT_TOK - 1) / QT_TOK, H, 3);
    int32_t* err = const_cast<int32_t*>(&st->dev_error);
    const int rows_tok = (L.hs == D && Dp == D) ? (QT_TOK + H - 1) / H : 0;
    quant_kernel<<<grid, QT_THREADS, 0, s>>>(st, q, k, v, L, cu, nseq, T, H, D, Dp, q8, k8, v8t, Tv,
                                             err, rows_tok);
    return cudaGetLastError();
}

}  // namespace vitfp8
