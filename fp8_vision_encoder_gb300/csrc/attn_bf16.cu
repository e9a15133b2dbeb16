// BF16 variable-length non-causal attention: the comparison path.
//
// "FP8 ViT Encoder Attention", Performance: every table compares the FP8 path
// with BF16 attention on the same workload.  This kernel is the BF16 column,
// built like the FP8 kernel so the two differ only in the arithmetic: the same
// work items (256 queries of one segment and head), the same warp roles (TMA
// warp, one MMA issuer, two softmax warpgroups), P kept in tensor memory over
// S, S of the next key tile issued right after each tile's P.V.
//
// Differences from the FP8 kernel:
//   * tcgen05.mma kind::f16 (BF16 x BF16 -> F32), K = 16 per instruction;
//   * Q, K and V are read straight from the bf16 [T][H][D] tensors; a 128-d
//     row is two 128-byte swizzled blocks of 64 elements;
//   * V is the B operand in MN-major form (d contiguous), so no transpose;
//   * P = bf16(2^(x - m_ref)) occupies 64 TMEM columns; as in the FP8 kernel
//     the row sum adds the rounded weights, so the weights applied to V sum
//     to one; two K/V stages (the bf16 tiles are twice as large).
// Key tiles start at the segment start (no alignment constraint on the token
// coordinate here); keys outside the segment are masked.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

namespace fb {
constexpr int BM = 128;
constexpr int NQT = 2;
constexpr int ROWS_PER_ITEM = BM * NQT;
constexpr int BN = 128;
constexpr int NST = 2;
constexpr int NUM_THREADS = 320;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int BLK = 128 * 128;     // one 128-row x 128-byte swizzled block (64 bf16 per row)
constexpr int TILE = 2 * BLK;      // 128 rows x 128 bf16 = two blocks along d

constexpr int SM_Q = 0;                      // [NQT] tiles
constexpr int SM_K = SM_Q + NQT * TILE;      // [NST]
constexpr int SM_V = SM_K + NST * TILE;      // [NST]: V rows are keys, blocks split d
constexpr int SM_BAR = SM_V + NST * TILE;
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_VFULL = B_KFULL + NST;
constexpr int B_KVEMPTY = B_VFULL + NST;
constexpr int B_SFULL = B_KVEMPTY + NST;
constexpr int B_PFULL = B_SFULL + NQT;
constexpr int B_OREADY = B_PFULL + NQT;
constexpr int B_FINAL = B_OREADY + NQT;
constexpr int NBAR = B_FINAL + 1;
constexpr int SM_TMEMPTR = SM_BAR + NBAR * 8;
constexpr int SM_ABORT = SM_TMEMPTR + 4;
constexpr int SM_USED = SM_ABORT + 4;
constexpr int SMEM_BYTES = SM_USED + 1024;
constexpr uint32_t TMEM_COLS = 512;
}  // namespace fb

__global__ void __launch_bounds__(fb::NUM_THREADS, 1)
attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace fb;
    const int item = blockIdx.x;
    const int total = p.ws->total_items;
    if (item >= total) return;

    int lo = 0, hi = p.nseq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int b = p.order[lo];
    const int local = item - p.prefix[lo];
    const int seg_s = p.cu[b];
    const int seg_e = p.cu[b + 1];
    const int L = seg_e - seg_s;
    const int nq = (L + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
    const int h = local / nq;
    const int qt = local - h * nq;
    const int q0 = seg_s + qt * ROWS_PER_ITEM;
    const int kbase = seg_s;
    const int nkv = (seg_e - kbase + BN - 1) / BN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);
    int32_t* err = &p.ws->error;
    auto BAR = [&](int i) -> uint32_t { return sb + SM_BAR + 8u * uint32_t(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_KVEMPTY + s), 1);
        }
        for (int w = 0; w < NQT; ++w) {
            mbar_init(BAR(B_SFULL + w), 1);
            mbar_init(BAR(B_PFULL + w), 4);
            mbar_init(BAR(B_OREADY + w), 1);
        }
        mbar_init(BAR(B_FINAL), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(sb + SM_TMEMPTR, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEMPTR);

    if (warp == WARP_TMA) {
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            // d 64..127 only when the head has them (a box wholly past D is skipped)
            const int nblk = p.D > 64 ? 2 : 1;
            mbar_arrive_expect_tx(BAR(B_QFULL), NQT * nblk * BLK);
            for (int w = 0; w < NQT; ++w)
                for (int blk = 0; blk < nblk; ++blk)
                    tma_load_3d(sb + SM_Q + w * TILE + blk * BLK, &tmQ, BAR(B_QFULL), blk * 64, h,
                                q0 + w * BM);
            int j = 0;
            for (; j < nkv; ++j) {
                const int s = j % NST;
                if (j >= NST && !bwait(BAR(B_KVEMPTY + s), ((j / NST) - 1) & 1, abort_flag, err)) break;
                const int key0 = kbase + j * BN;
                mbar_arrive_expect_tx(BAR(B_KFULL + s), nblk * BLK);
                for (int blk = 0; blk < nblk; ++blk)
                    tma_load_3d(sb + SM_K + s * TILE + blk * BLK, &tmK, BAR(B_KFULL + s), blk * 64, h, key0);
                mbar_arrive_expect_tx(BAR(B_VFULL + s), nblk * BLK);
                for (int blk = 0; blk < nblk; ++blk)
                    tma_load_3d(sb + SM_V + s * TILE + blk * BLK, &tmV, BAR(B_VFULL + s), blk * 64, h, key0);
            }
            if (*abort_flag) {
                bwait(BAR(B_QFULL), 0, abort_flag, err);
                for (int jj = (j > NST ? j - NST : 0); jj < j; ++jj) {
                    const int s = jj % NST;
                    const uint32_t ph = (jj / NST) & 1;
                    for (int spin = 0; spin < (1 << 22); ++spin)
                        if (mbar_try_wait(BAR(B_KFULL + s), ph)) break;
                    for (int spin = 0; spin < (1 << 22); ++spin)
                        if (mbar_try_wait(BAR(B_VFULL + s), ph)) break;
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            const uint32_t idS = make_idesc(1, BM, BN);
            const uint32_t idPV = make_idesc_bmn(1, BM, p.DV);
            const uint64_t dQ[NQT] = {sw128_kmajor_desc(sb + SM_Q), sw128_kmajor_desc(sb + SM_Q + TILE)};
            const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
            // V: MN-major (d contiguous), 64-element d groups BLK apart, 8-key
            // groups 1024 bytes apart; one K step (16 keys) advances 2048 bytes.
            const uint64_t dV0 = sw128_mnmajor_desc(sb + SM_V, BLK, 1024);
            const int KS = (p.D + 15) / 16;  // 16-wide K steps over d
            auto issue_S = [&](int w, int s) {
                const uint64_t dk = dK0 + uint64_t(s * (TILE >> 4));
                const uint32_t dS = tmem + uint32_t(w * 128);
                for (int kk = 0; kk < KS; ++kk) {
                    // step kk: block kk / 4, 32-byte offset (kk % 4) inside the row
                    const uint64_t off = uint64_t((kk >> 2) * (BLK >> 4) + 2 * (kk & 3));
                    umma_bf16(dS, dQ[w] + off, dk + off, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(B_SFULL + w));
            };
            bool ok = bwait(BAR(B_QFULL), 0, abort_flag, err) &&
                      bwait(BAR(B_KFULL + 0), 0, abort_flag, err);
            if (ok) {
                tc_fence_after();
                issue_S(0, 0);
                issue_S(1, 0);
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const int s = j % NST;
                const uint32_t ph = (j / NST) & 1;
                const bool nxt = j + 1 < nkv;
                const int s1 = (j + 1) % NST;
                const uint32_t ph1 = ((j + 1) / NST) & 1;
                if (!(ok = bwait(BAR(B_VFULL + s), ph, abort_flag, err))) break;
                if (nxt && !(ok = bwait(BAR(B_KFULL + s1), ph1, abort_flag, err))) break;
                const uint64_t dv = dV0 + uint64_t(s * (TILE >> 4));
                for (int w = 0; w < NQT; ++w) {
                    if (!(ok = bwait(BAR(B_PFULL + w), j & 1, abort_flag, err))) break;
                    tc_fence_after();
                    const uint32_t dO = tmem + uint32_t(256 + w * 128);
                    const uint32_t aP = tmem + uint32_t(w * 128);
                    // K = 128 keys in 8 steps of 16: P columns + 8, V + 2048 bytes
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_bf16_ts(dO, aP + uint32_t(8 * kk), dv + uint64_t(kk * (2048 >> 4)), idPV,
                                     (j > 0 || kk > 0) ? 1u : 0u);
                    if (nxt)
                        issue_S(w, s1);
                    else
                        tc_commit(BAR(B_OREADY + w));
                }
                if (!ok) break;
                tc_commit(BAR(B_KVEMPTY + s));
            }
            tc_commit(BAR(B_FINAL));
            for (int spin = 0; spin < (1 << 24); ++spin)
                if (mbar_try_wait(BAR(B_FINAL), 0)) break;
        }
    } else if (warp < 8) {
        const int w = warp >> 2;
        const int sub = warp & 3;
        const int r = sub * 32 + lane;
        const int qrow = q0 + w * BM + r;
        const bool row_valid = qrow < seg_e;
        const uint32_t lane_off = uint32_t(sub * 32) << 16;
        const uint32_t tS = tmem + lane_off + uint32_t(w * 128);
        const uint32_t tO = tmem + lane_off + uint32_t(256 + w * 128);
        const float c = p.sm_scale * 1.4426950408889634f;
        float m_ref = 0.0f;
        float l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_SFULL + w), j & 1, abort_flag, err));
            if (!ok) break;
            tc_fence_after();
            uint32_t s0[32], s1[32], s2[32], s3[32];
            tmem_ld_32x32b_x32(tS + 0, s0);
            tmem_ld_32x32b_x32(tS + 32, s1);
            tmem_ld_32x32b_x32(tS + 64, s2);
            tmem_ld_32x32b_x32(tS + 96, s3);
            tmem_ld_wait(s0);
            reg_fence32(s1);
            reg_fence32(s2);
            reg_fence32(s3);
            float sf[128];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                sf[i] = __uint_as_float(s0[i]);
                sf[32 + i] = __uint_as_float(s1[i]);
                sf[64 + i] = __uint_as_float(s2[i]);
                sf[96 + i] = __uint_as_float(s3[i]);
            }
            const int key0 = kbase + j * BN;
            if (key0 + BN > seg_e) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (key0 + i >= seg_e) sf[i] = -INFINITY;
            }
            float mx0 = sf[0], mx1 = sf[1], mx2 = sf[2], mx3 = sf[3];
#pragma unroll
            for (int i = 4; i < 128; i += 8) {
                mx0 = fmax3(mx0, sf[i], sf[i + 1]);
                mx1 = fmax3(mx1, sf[i + 2], sf[i + 3]);
                mx2 = fmax3(mx2, sf[i + 4], sf[i + 5]);
                mx3 = fmax3(mx3, sf[i + 6], sf[i + 7]);
            }
            const float xmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
            float oscale = 1.0f;
            bool need = false;
            if (j == 0) {
                m_ref = ceilf(xmax);
            } else if (xmax > m_ref) {
                const float mnew = ceilf(xmax);
                oscale = exp2_int(m_ref - mnew);
                l *= oscale;
                m_ref = mnew;
                need = true;
            }
            const float bias = -m_ref;
            // P (bf16) into the first 64 columns of S: keys 0..63 in columns
            // 0..31, keys 64..127 in 32..63, two keys per column (lower key
            // in the low half).  Each half is stored as soon as it is packed.
            float ls = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
                float la = 0.f, lb = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float a0 = ex2_approx(fmaf(sf[64 * half + 2 * i], c, bias));
                    const float a1 = ex2_approx(fmaf(sf[64 * half + 2 * i + 1], c, bias));
                    pk[i] = cvt_bf16x2(a0, a1);
                    // the row sum adds the weights as rounded (bf16 -> f32 is exact)
                    const float r0 = __uint_as_float(pk[i] << 16);
                    const float r1 = __uint_as_float(pk[i] & 0xFFFF0000u);
                    if (i & 1) lb += r0 + r1; else la += r0 + r1;
                }
                ls += la + lb;
                tmem_st_32x32b_x32(tS + uint32_t(32 * half), pk);
            }
            l += ls;
            if (__any_sync(0xFFFFFFFFu, need)) {
                for (int cc = 0; cc < p.DV; cc += 16) {
                    uint32_t o[16];
                    tmem_ld_32x32b_x16(tO + uint32_t(cc), o);
                    tmem_ld_wait16(o);
#pragma unroll
                    for (int q = 0; q < 16; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * oscale);
                    tmem_st_32x32b_x16(tO + uint32_t(cc), o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_PFULL + w));
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OREADY + w), 0, abort_flag, err));
        if (ok) {
            tc_fence_after();
            const float oscale = 1.0f / l;
            uint16_t* orow = p.out + (int64_t(qrow) * p.H + h) * p.D;
            for (int cc = 0; cc < p.DV; cc += 16) {
                uint32_t o[16];
                tmem_ld_32x32b_x16(tO + uint32_t(cc), o);
                tmem_ld_wait16(o);
                uint32_t pkd[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    pkd[q] = cvt_bf16x2(__uint_as_float(o[2 * q]) * oscale, __uint_as_float(o[2 * q + 1]) * oscale);
                if (row_valid) {
                    if (cc + 8 <= p.D)
                        *reinterpret_cast<uint4*>(orow + cc) = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
                    if (cc + 16 <= p.D)
                        *reinterpret_cast<uint4*>(orow + cc + 8) = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

namespace {
using EncodeFnB = decltype(&cuTensorMapEncodeTiled);

EncodeFnB get_encode_fn_b() {
    static EncodeFnB fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFnB>(ptr);
    }
    return fn;
}

// bf16 [T][H][D] with token stride H*D: box 64 d x 1 head x 128 tokens.
bool make_map_bf16(CUtensorMap* m, const void* base, int T, int H, int D) {
    auto enc = get_encode_fn_b();
    if (!enc) return false;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(T)};
    cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(H) * D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

vitfp8_status launch_attn_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* cu, int nseq, int T, int H, int D, float sm_scale,
                               uint16_t* out, void* ws, cudaStream_t s) {
    using namespace fb;
    CUtensorMap mq, mk, mv;
    if (!make_map_bf16(&mq, q, T, H, D) || !make_map_bf16(&mk, k, T, H, D) ||
        !make_map_bf16(&mv, v, T, H, D))
        return VITFP8_ERR_CUDA;
    if (launch_attn_plan(cu, nseq, T, H, ROWS_PER_ITEM, ws, s) != cudaSuccess) return VITFP8_ERR_CUDA;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES) != cudaSuccess)
            return VITFP8_ERR_CUDA;
        attr_set = true;
    }
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    AttnParams prm;
    prm.cu = cu;
    prm.order = reinterpret_cast<const int32_t*>(hdr + 1);
    prm.prefix = prm.order + nseq;
    prm.ws = hdr;
    prm.st = nullptr;
    prm.out = out;
    prm.nseq = nseq;
    prm.T = T;
    prm.H = H;
    prm.D = D;
    prm.DV = (D + 15) & ~15;
    prm.KS = (D + 15) / 16;
    prm.sm_scale = sm_scale;
    const long long grid = (long long)((T + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM + nseq) * H;
    if (grid > 0x7FFFFFFFLL) return VITFP8_ERR_UNSUPPORTED;
    attn_bf16_kernel<<<unsigned(grid), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

}  // namespace vitfp8
