// BF16 variable-length non-causal attention: the comparison path.
//
// "FP8 ViT Encoder Attention", Performance: every table compares the FP8 path
// with BF16 attention on the same workload.  This kernel is the BF16 column,
// built like the FP8 kernel so that the two differ in the arithmetic and in
// what the arithmetic forces:
//
//   * one CTA: one query tile of 128 rows against every key tile of its
//     segment; warp 8 loads (TMA), warp 9 issues S = Q K^T, warp 10 issues
//     O += P V, warps 0-7 run the softmax with two threads of one warp per row
//     (TMEM access shape 16x32bx2) and the row maximum returned by the score
//     load (tcgen05.ld.red);
//   * tcgen05.mma kind::f16 (BF16 x BF16 -> F32), K = 16 per instruction, so
//     a key tile of 128 costs the tensor core as much as 256 keys in FP8: the
//     key tiles are 128 wide, and S and P are both double-buffered in TMEM
//     (S 2 x 128 columns, O 128, P 2 x 64: bf16 pairs), which lets S(j+1) run
//     while the softmax works on S(j) and decouples the softmax warps;
//   * Q, K and V are read straight from the bf16 [T][H][D] tensors, a 128-d
//     row being two 128-byte swizzled blocks of 64 elements; V is the B
//     operand in MN-major form (d contiguous), so no transpose is needed;
//   * P = bf16(2^(x - m_ref)) and l is the fp32 sum of those rounded weights
//     (the weights applied to V sum to one), computed by the softmax threads.
//
// Key tiles start at the segment start (no alignment constraint on the token
// coordinate); keys outside the segment are masked.  Every wait is bounded.
//
// As on the FP8 path, attn_bf16_persistent_kernel runs the same roles and the
// same softmax tile (softmax_tile_bf16) with one CTA per SM walking the work
// items, for segments of up to 6144 tokens; the outputs are bit-identical.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "host_once.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

namespace fb {
constexpr int BM = 128;                  // query rows per CTA
constexpr int ROWS_PER_ITEM = BM;
constexpr int BN = 128;                  // keys per tile
constexpr int HALF = BN / 2;             // keys per softmax thread and tile
constexpr int NST = 3;                   // K/V pipeline stages
constexpr int NUM_THREADS = 352;         // 8 softmax warps, TMA warp, S and P.V issuers
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;              // S issuer; owns the TMEM allocation
constexpr int WARP_PV = 10;              // P.V issuer
constexpr int BLK = 128 * 128;           // one 128-row x 128-byte swizzled block (64 bf16 per row)
constexpr int TILE = 2 * BLK;            // 128 rows x 128 bf16 = two blocks along d

constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + TILE;
constexpr int SM_V = SM_K + NST * TILE;  // V rows are keys, blocks split d
constexpr int SM_BAR = SM_V + NST * TILE;
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_VFULL = B_KFULL + NST;
constexpr int B_KEMPTY = B_VFULL + NST;
constexpr int B_VEMPTY = B_KEMPTY + NST;
constexpr int B_SFULL = B_VEMPTY + NST;  // [2]: S(j) in buffer j%2 complete
constexpr int B_SFREE = B_SFULL + 2;     // [2]: S(j) read by all 8 softmax warps
constexpr int B_PFULL = B_SFREE + 2;     // [2]: P(j) written by all 8 softmax warps
constexpr int B_OFULL = B_PFULL + 2;     // [2]: P(j) V_j (and every earlier P.V) complete
constexpr int B_FINAL = B_OFULL + 2;
constexpr int B_QEMPTY = B_FINAL + 1;    // persistent: every S product of the unit is done with Q
constexpr int B_OFREE = B_QEMPTY + 1;    // persistent: the 8 softmax warps have read the unit's O
constexpr int B_IFULL = B_OFREE + 1;     // persistent [2]: work-unit description written
constexpr int B_IEMPTY = B_IFULL + 2;    // persistent [2]: description used up by all 10 consumers
constexpr int NBAR = B_IEMPTY + 2;
constexpr int IEMPTY_COUNT = 10;         // S issuer, P.V issuer, 8 softmax warps
constexpr int SM_TMEMPTR = SM_BAR + NBAR * 8;
constexpr int SM_ABORT = SM_TMEMPTR + 4;
constexpr int SM_INFO = SM_ABORT + 4;    // persistent: 2 descriptions of INFO_INTS ints
constexpr int INFO_INTS = 8;
constexpr int I_WORK = 0, I_H = 1, I_Q0 = 2, I_SEGS = 3, I_SEGE = 4, I_NKV = 5;
constexpr int SM_USED = SM_INFO + 2 * INFO_INTS * 4;
constexpr int SMEM_BYTES = SM_USED + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 384;   // S and P: buffer b at + b * 128 / + b * 64
constexpr int OSPLIT = 64;               // O columns per half-row thread
constexpr float RESCALE_AT = 8.0f;       // the reference moves when P would exceed 2^8
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
}  // namespace fb

// Softmax of one 128-key tile, shared by both BF16 kernels (the 8 softmax
// warps, two threads per row): wait for S in buffer g % 2, read it with its
// 32-key chunk maxima, mask keys past the segment, move the reference when
// needed (O and l rescaled by an exact power of two), write P = bf16(2^(x -
// m_ref)) into P buffer g % 2 and add the rounded weights to l.  g counts
// tiles (across work units in the persistent kernel); first marks a unit's
// first tile; key0 is this thread's first key.  False when a wait gave up.
struct SoftmaxWarpB {
    uint32_t tmem, lane_off, tO;
    uint32_t bar0;            // shared-memory address of barrier 0
    uint64_t c2;
    float c;
    volatile int* abort_flag;
    int32_t* err;
};

__device__ __forceinline__ bool softmax_tile_bf16(const SoftmaxWarpB& x, uint32_t g, int key0, int seg_e,
                                                  bool first, float& m_ref, float& l) {
    using namespace fb;
    const int lane = threadIdx.x & 31;
    auto BAR = [&](int i) -> uint32_t { return x.bar0 + 8u * uint32_t(i); };
    const int sbuf = int(g & 1u);
    if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_SFULL + sbuf), (g >> 1) & 1u, x.abort_flag, x.err))) return false;
    tc_fence_after();
    const uint32_t tS = x.tmem + x.lane_off + TM_S + uint32_t(sbuf * BN);
    float s0[32], s1[32];
    float m0, m1;
    tmem_ld_16x2_x32_max<HALF>(tS + 0, s0, m0);
    tmem_ld_16x2_x32_max<HALF>(tS + 32, s1, m1);
    tmem_ld_wait_f32(s0);
    reg_fence_f32(s1);
    asm volatile("" : "+f"(m0), "+f"(m1));
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_SFREE + sbuf));

    float sf[HALF];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        sf[i] = s0[i];
        sf[32 + i] = s1[i];
    }
    float pmax = fmaxf(m0, m1);
    if (key0 + HALF > seg_e) {
        // Last tile: keys past the segment are masked.
#pragma unroll
        for (int i = 0; i < HALF; ++i)
            if (key0 + i >= seg_e && VF_IN(i, 1, HALF, x.err)) sf[i] = -INFINITY;
        float mx0 = sf[0], mx1 = sf[1];
#pragma unroll
        for (int i = 2; i + 4 <= HALF; i += 4) {
            mx0 = fmax3(mx0, sf[i], sf[i + 1]);
            mx1 = fmax3(mx1, sf[i + 2], sf[i + 3]);
        }
        mx0 = fmax3(mx0, sf[HALF - 2], sf[HALF - 1]);
        pmax = fmaxf(mx0, mx1);
    }
    pmax = fmaxf(pmax, __shfl_xor_sync(0xFFFFFFFFu, pmax, 16));
    const float xmax = pmax * x.c;
    float oscale = 1.0f;
    bool need = false;
    if (first) {
        m_ref = ceilf(xmax);
    } else if (xmax > m_ref + RESCALE_AT) {
        // bf16 and fp32 have range to spare: the reference moves only
        // when P would pass 2^8.
        const float mnew = ceilf(xmax);
        oscale = exp2_int(m_ref - mnew);
        l *= oscale;
        m_ref = mnew;
        need = true;
    }
    const uint64_t b2 = f32x2_pack(-m_ref, -m_ref);
    // P = bf16(2^(x - m_ref)), two keys per 32-bit word (lower key in the
    // low half); l adds the rounded weights (bf16 -> f32 is exact).
    uint32_t pk[HALF / 2];
    float la = 0.f, lb = 0.f;
#pragma unroll
    for (int q = 0; q < HALF / 2; ++q) {
        float y0, y1;
        f32x2_unpack(ffma2(f32x2_pack(sf[2 * q], sf[2 * q + 1]), x.c2, b2), y0, y1);
        pk[q] = cvt_bf16x2(ex2_approx(y0), ex2_approx(y1));
        const float r0 = __uint_as_float(pk[q] << 16);
        const float r1 = __uint_as_float(pk[q] & 0xFFFF0000u);
        if (q & 1) lb += r0 + r1; else la += r0 + r1;
    }
    l += la + lb;

    const int pb = sbuf;
    if (__any_sync(0xFFFFFFFFu, need)) {
        // O must hold every P.V before this tile: wait for the previous one.
        if (!__all_sync(0xFFFFFFFFu,
                        bwait(BAR(B_OFULL + (pb ^ 1)), ((g - 1u) >> 1) & 1u, x.abort_flag, x.err)))
            return false;
        tc_fence_after();
        const uint64_t s2v = f32x2_pack(oscale, oscale);
        uint32_t oa[32], ob[32];
        tmem_ld_16x2_x32<OSPLIT>(x.tO + 0u, oa);
        tmem_ld_16x2_x32<OSPLIT>(x.tO + 32u, ob);
        tmem_ld_wait(oa);
        reg_fence32(ob);
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
            float a0, a1;
            f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(oa[q]), __uint_as_float(oa[q + 1])), s2v), a0, a1);
            oa[q] = __float_as_uint(a0);
            oa[q + 1] = __float_as_uint(a1);
            f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(ob[q]), __uint_as_float(ob[q + 1])), s2v), a0, a1);
            ob[q] = __float_as_uint(a0);
            ob[q + 1] = __float_as_uint(a1);
        }
        tmem_st_16x2_x32<OSPLIT>(x.tO + 0u, oa);
        tmem_st_16x2_x32<OSPLIT>(x.tO + 32u, ob);
    }
    if (g >= 2u) {
        // P buffer g % 2 is free once the P.V two tiles back is complete.
        if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL + pb), ((g - 2u) >> 1) & 1u, x.abort_flag, x.err)))
            return false;
        tc_fence_after();
    }
    // This half of the P row: 64 keys in 32 columns (lanes 16-31 at +32).
    tmem_st_16x2_x32<HALF / 2>(x.tmem + x.lane_off + TM_P + uint32_t(pb * (BN / 2)), pk);
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_PFULL + pb));
    return true;
}

__global__ void __launch_bounds__(fb::NUM_THREADS, 1)
attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace fb;
    const int item = blockIdx.x;
    SegRec rec;
    int total;
    if (!find_item(p, item, rec, total) || item >= total) return;
    const int local = item - rec.first_item;
    const int seg_s = rec.seg_s;
    const int seg_e = rec.seg_e;
    const int nq = rec.nq;
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
            mbar_init(BAR(B_KEMPTY + s), 1);
            mbar_init(BAR(B_VEMPTY + s), 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(BAR(B_SFULL + b2), 1);
            mbar_init(BAR(B_SFREE + b2), 8);
            mbar_init(BAR(B_PFULL + b2), 8);
            mbar_init(BAR(B_OFULL + b2), 1);
        }
        mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
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
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            // d 64..127 only when the head has them (a box wholly past D is skipped)
            const int nblk = p.D > 64 ? 2 : 1;
            mbar_arrive_expect_tx(BAR(B_QFULL), nblk * BLK);
            for (int blk = 0; blk < nblk; ++blk)
                tma_load_3d(sb + SM_Q + blk * BLK, &tmQ, BAR(B_QFULL), blk * 64, h, q0);
            int j = 0;
            for (; j < nkv; ++j) {
                const int s = j % NST;
                const int key0 = kbase + j * BN;
                if (j >= NST && !bwait(BAR(B_KEMPTY + s), ((j / NST) - 1) & 1, abort_flag, err)) break;
                mbar_arrive_expect_tx(BAR(B_KFULL + s), nblk * BLK);
                for (int blk = 0; blk < nblk; ++blk)
                    tma_load_3d(sb + SM_K + s * TILE + blk * BLK, &tmK, BAR(B_KFULL + s), blk * 64, h, key0);
                if (j >= NST && !bwait(BAR(B_VEMPTY + s), ((j / NST) - 1) & 1, abort_flag, err)) {
                    ++j;   // K_j is in flight: its barrier is drained below
                    break;
                }
                mbar_arrive_expect_tx(BAR(B_VFULL + s), nblk * BLK);
                for (int blk = 0; blk < nblk; ++blk)
                    tma_load_3d(sb + SM_V + s * TILE + blk * BLK, &tmV, BAR(B_VFULL + s), blk * 64, h, key0);
            }
            if (*abort_flag) {
                // Let the copies this thread started land before the CTA exits.
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
        // ------------------------------------------------ S issuer
        if (lane == 0) {
            const uint32_t idS = make_idesc(1, BM, BN);
            const uint64_t dQ = sw128_kmajor_desc(sb + SM_Q);
            const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
            const int KS = (p.D + 15) / 16;  // 16-wide K steps over d
            bool ok = bwait(BAR(B_QFULL), 0, abort_flag, err);
            int s = 0;
            uint32_t ph = 0;
            for (int t = 0; ok && t < nkv; ++t) {
                // S(t) into buffer t % 2 once K_t is in and S(t-2) has been read.
                const int sbuf = t & 1;
                if (!(ok = bwait(BAR(B_KFULL + s), ph, abort_flag, err))) break;
                if (t >= 2 && !(ok = bwait(BAR(B_SFREE + sbuf), ((t - 2) >> 1) & 1, abort_flag, err))) break;
                tc_fence_after();
                const uint64_t dk = dK0 + uint64_t(s * (TILE >> 4));
                const uint32_t dS = tmem + TM_S + uint32_t(sbuf * BN);
                for (int kk = 0; kk < KS; ++kk) {
                    // step kk: block kk / 4, 32-byte offset (kk % 4) inside the row
                    const uint64_t off = uint64_t((kk >> 2) * (BLK >> 4) + 2 * (kk & 3));
                    umma_bf16(dS, dQ + off, dk + off, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(BAR(B_SFULL + sbuf));
                tc_commit(BAR(B_KEMPTY + s));
                if (++s == NST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // Every MMA issued above has completed before TMEM is released.
            tc_commit(BAR(B_FINAL));
            for (int spin = 0; spin < (1 << 24); ++spin)
                if (mbar_try_wait(BAR(B_FINAL), 0)) break;
        }
    } else if (warp == WARP_PV) {
        // ------------------------------------------------ P.V issuer
        if (lane == 0) {
            const uint32_t idPV = make_idesc_bmn(1, BM, p.DV);
            // V: MN-major (d contiguous), 64-element d groups BLK apart, 8-key
            // groups 1024 bytes apart; one K step (16 keys) advances 2048 bytes.
            const uint64_t dV0 = sw128_mnmajor_desc(sb + SM_V, BLK, 1024);
            const uint32_t tO = tmem + TM_O;
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int j = 0; ok && j < nkv; ++j) {
                const int pb = j & 1;
                if (!(ok = bwait(BAR(B_VFULL + s), ph, abort_flag, err))) break;
                if (!(ok = bwait(BAR(B_PFULL + pb), (j >> 1) & 1, abort_flag, err))) break;
                tc_fence_after();
                const uint32_t aP = tmem + TM_P + uint32_t(pb * (BN / 2));
                const uint64_t dv = dV0 + uint64_t(s * (TILE >> 4));
                // K = 128 keys in 8 steps of 16: P columns + 8, V + 2048 bytes
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_bf16_ts(tO, aP + uint32_t(8 * kk), dv + uint64_t(kk * (2048 >> 4)), idPV,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(B_OFULL + pb));
                tc_commit(BAR(B_VEMPTY + s));
                if (++s == NST) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            tc_commit(BAR(B_FINAL));
            for (int spin = 0; spin < (1 << 24); ++spin)
                if (mbar_try_wait(BAR(B_FINAL), 0)) break;
        }
    } else if (warp < 8) {
        // ------------------------------------------------ softmax (warps 0..7)
        const int half = lane >> 4;           // keys half*64 .. half*64+63 of each tile
        const int rbase = 32 * (warp & 3) + 16 * (warp >> 2);
        const int r = rbase + (lane & 15);    // row inside the query tile
        const int qrow = q0 + r;
        const bool row_valid = qrow < seg_e;
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tO = tmem + lane_off + TM_O;
        const float c = p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        float m_ref = 0.0f;
        float l = 0.0f;
        bool ok = true;
        const SoftmaxWarpB sw{tmem, lane_off, tO, sb + SM_BAR, c2, c, abort_flag, err};
        for (int j = 0; j < nkv; ++j) {
            ok = softmax_tile_bf16(sw, uint32_t(j), kbase + j * BN + half * HALF, seg_e, j == 0, m_ref, l);
            if (!ok) break;
        }
        if (ok)
            ok = __all_sync(0xFFFFFFFFu,
                            bwait(BAR(B_OFULL + ((nkv - 1) & 1)), ((nkv - 1) >> 1) & 1, abort_flag, err));
        if (ok) {
            tc_fence_after();
            const float oscale = 1.0f / (l + __shfl_xor_sync(0xFFFFFFFFu, l, 16));
            uint16_t* orow = p.out + (int64_t(qrow) * p.H + h) * p.D;
            for (int cc = 0; cc < OSPLIT; cc += 16) {
                uint32_t o[16];
                tmem_ld_16x2_x16<OSPLIT>(tO + uint32_t(cc), o);
                tmem_ld_wait16(o);
                uint32_t pkd[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    pkd[q] = cvt_bf16x2(__uint_as_float(o[2 * q]) * oscale, __uint_as_float(o[2 * q + 1]) * oscale);
                const int d0 = half * OSPLIT + cc;
                if (row_valid) {
                    [[maybe_unused]] const int64_t o0 = (int64_t(qrow) * p.H + h) * p.D + d0;   // checked build
                    if (d0 + 8 <= p.D && VF_IN(o0, 8, p.out_elems, err))
                        *reinterpret_cast<uint4*>(orow + d0) = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
                    if (d0 + 16 <= p.D && VF_IN(o0 + 8, 8, p.out_elems, err))
                        *reinterpret_cast<uint4*>(orow + d0 + 8) = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
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

// The same roles over many work items per CTA (one CTA per SM), for short
// segments: the TMA warp takes items from the call's counter, publishes each
// in a two-slot description ring and loads its Q and K/V tiles while the
// previous item finishes.  S and P buffers, ring stages and barrier phases
// count tiles across items (g); an item's first P.V waits for the softmax to
// have read the previous item's O.  Same arithmetic per item as
// attn_bf16_kernel, so the outputs are bit-identical.
__global__ void __launch_bounds__(fb::NUM_THREADS, 1)
attn_bf16_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace fb;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);
    int32_t* err = &p.ws->error;
    auto BAR = [&](int i) -> uint32_t { return sb + SM_BAR + 8u * uint32_t(i); };
    auto INFO = [&](int slot) -> volatile int* {
        return reinterpret_cast<volatile int*>(smem + SM_INFO + slot * INFO_INTS * 4);
    };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nblk = p.D > 64 ? 2 : 1;   // d 64..127 only when the head has them

    // An item -> (head, query rows, segment, key tiles), decoded by the whole
    // TMA warp (one vote over the records).
    struct Item { int h, q0, seg_s, seg_e, nkv; };
    int4 mine = make_int4(0, 0, 0, 0);
    int total = 0;
    auto decode = [&](int item, Item& w) -> bool {
        SegRec rec;
        if (!find_item_pick(p, item, mine, rec)) return false;
        const int local = item - rec.first_item;
        w.h = local / rec.nq;
        w.q0 = rec.seg_s + (local - w.h * rec.nq) * ROWS_PER_ITEM;
        w.seg_s = rec.seg_s;
        w.seg_e = rec.seg_e;
        w.nkv = (rec.seg_e - rec.seg_s + BN - 1) / BN;
        return true;
    };
    auto publish = [&](int slot, bool have, const Item& w) {
        volatile int* inf = INFO(slot);
        inf[I_WORK] = have ? 1 : 0;
        if (have) {
            inf[I_H] = w.h;
            inf[I_Q0] = w.q0;
            inf[I_SEGS] = w.seg_s;
            inf[I_SEGE] = w.seg_e;
            inf[I_NKV] = w.nkv;
        }
        mbar_arrive(BAR(B_IFULL + slot));
    };
    Item w0;
    bool have0 = false;
    if (warp == WARP_TMA) {
        mine = find_item_load(p);
        total = p.ws->total_items;
        have0 = int(blockIdx.x) < total && decode(blockIdx.x, w0);
        if (lane == 0) {
            mbar_init(BAR(B_QFULL), 1);
            for (int s = 0; s < NST; ++s) {
                mbar_init(BAR(B_KFULL + s), 1);
                mbar_init(BAR(B_VFULL + s), 1);
                mbar_init(BAR(B_KEMPTY + s), 1);
                mbar_init(BAR(B_VEMPTY + s), 1);
            }
            for (int b2 = 0; b2 < 2; ++b2) {
                mbar_init(BAR(B_SFULL + b2), 1);
                mbar_init(BAR(B_SFREE + b2), 8);
                mbar_init(BAR(B_PFULL + b2), 8);
                mbar_init(BAR(B_OFULL + b2), 1);
                mbar_init(BAR(B_IFULL + b2), 1);
                mbar_init(BAR(B_IEMPTY + b2), IEMPTY_COUNT);
            }
            mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
            mbar_init(BAR(B_QEMPTY), 1);
            mbar_init(BAR(B_OFREE), 8);
            *abort_flag = 0;
            fence_mbar_init();
            publish(0, have0, w0);
        }
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
        // ------------------------------------------------ TMA producer
        int g = 0;            // K/V tiles whose copies were started (K and V)
        int kq = 0;           // Q tiles started
        bool k_only = false;  // K of tile g started, its V not
        bool ok = true;
        Item w = w0;
        bool have = have0;
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        for (int qi = 0; ok && have; ++qi) {
            if (lane == 0) {
                const int slot = qi & 1;
                if (qi > 0) {
                    if (qi >= 2) ok = bwait(BAR(B_IEMPTY + slot), ((qi - 2) >> 1) & 1, abort_flag, err);
                    if (ok) publish(slot, true, w);
                }
                // Q of this item once every S product of the previous one is done.
                if (ok && qi > 0) ok = bwait(BAR(B_QEMPTY), (qi - 1) & 1, abort_flag, err);
                if (ok) {
                    mbar_arrive_expect_tx(BAR(B_QFULL), nblk * BLK);
                    for (int blk = 0; blk < nblk; ++blk)
                        tma_load_3d(sb + SM_Q + blk * BLK, &tmQ, BAR(B_QFULL), blk * 64, w.h, w.q0);
                    ++kq;
                }
                for (int j = 0; ok && j < w.nkv; ++j, ++g) {
                    const int s = g % NST;
                    const int key0 = w.seg_s + j * BN;
                    if (g >= NST && !(ok = bwait(BAR(B_KEMPTY + s), ((g / NST) - 1) & 1, abort_flag, err))) break;
                    mbar_arrive_expect_tx(BAR(B_KFULL + s), nblk * BLK);
                    for (int blk = 0; blk < nblk; ++blk)
                        tma_load_3d(sb + SM_K + s * TILE + blk * BLK, &tmK, BAR(B_KFULL + s), blk * 64, w.h, key0);
                    if (g >= NST && !(ok = bwait(BAR(B_VEMPTY + s), ((g / NST) - 1) & 1, abort_flag, err))) {
                        k_only = true;
                        break;
                    }
                    mbar_arrive_expect_tx(BAR(B_VFULL + s), nblk * BLK);
                    for (int blk = 0; blk < nblk; ++blk)
                        tma_load_3d(sb + SM_V + s * TILE + blk * BLK, &tmV, BAR(B_VFULL + s), blk * 64, w.h, key0);
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            int nu = 0;
            if (lane == 0) nu = int(gridDim.x) + atomicAdd(&p.ws->next_unit, 1);
            nu = __shfl_sync(0xFFFFFFFFu, nu, 0);
            have = nu < total && decode(nu, w);
            if (!have && lane == 0) {
                // "No more work" in the next slot, once it is free.
                const int slot = (qi + 1) & 1;
                if (qi + 1 < 2 || bwait(BAR(B_IEMPTY + slot), ((qi - 1) >> 1) & 1, abort_flag, err))
                    publish(slot, false, w);
            }
        }
        if (lane == 0 && *abort_flag) {
            // Let the copies this thread started land before the CTA exits.
            for (int spin = 0; spin < (1 << 22) && kq > 0; ++spin)
                if (mbar_try_wait(BAR(B_QFULL), (kq - 1) & 1)) break;
            const int gk = g + (k_only ? 1 : 0);
            for (int gg = (gk > NST ? gk - NST : 0); gg < gk; ++gg) {
                const int s = gg % NST;
                const uint32_t ph = (gg / NST) & 1;
                for (int spin = 0; spin < (1 << 22); ++spin)
                    if (mbar_try_wait(BAR(B_KFULL + s), ph)) break;
                for (int spin = 0; spin < (1 << 22) && gg < g; ++spin)
                    if (mbar_try_wait(BAR(B_VFULL + s), ph)) break;
            }
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ S issuer
        if (lane == 0) {
            const uint32_t idS = make_idesc(1, BM, BN);
            const uint64_t dQ = sw128_kmajor_desc(sb + SM_Q);
            const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
            const int KS = (p.D + 15) / 16;  // 16-wide K steps over d
            int s = 0;
            uint32_t ph = 0, g = 0;
            bool ok = true;
            for (int qi = 0; ok; ++qi) {
                const int slot = qi & 1;
                if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                if (!INFO(slot)[I_WORK]) break;
                const int nkv = INFO(slot)[I_NKV];
                if (!(ok = bwait(BAR(B_QFULL), qi & 1, abort_flag, err))) break;
                for (int j = 0; j < nkv; ++j, ++g) {
                    // S(g) into buffer g % 2 once K_g is in and S(g-2) has been read.
                    const int sbuf = int(g & 1u);
                    if (!(ok = bwait(BAR(B_KFULL + s), ph, abort_flag, err))) break;
                    if (g >= 2u && !(ok = bwait(BAR(B_SFREE + sbuf), ((g - 2u) >> 1) & 1u, abort_flag, err))) break;
                    tc_fence_after();
                    const uint64_t dk = dK0 + uint64_t(s * (TILE >> 4));
                    const uint32_t dS = tmem + TM_S + uint32_t(sbuf * BN);
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint64_t off = uint64_t((kk >> 2) * (BLK >> 4) + 2 * (kk & 3));
                        umma_bf16(dS, dQ + off, dk + off, idS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(BAR(B_SFULL + sbuf));
                    tc_commit(BAR(B_KEMPTY + s));
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(BAR(B_QEMPTY));   // every S product of this item read Q
                mbar_arrive(BAR(B_IEMPTY + slot));
            }
            tc_commit(BAR(B_FINAL));
            for (int spin = 0; spin < (1 << 24); ++spin)
                if (mbar_try_wait(BAR(B_FINAL), 0)) break;
        }
    } else if (warp == WARP_PV) {
        // ------------------------------------------------ P.V issuer
        if (lane == 0) {
            const uint32_t idPV = make_idesc_bmn(1, BM, p.DV);
            const uint64_t dV0 = sw128_mnmajor_desc(sb + SM_V, BLK, 1024);
            const uint32_t tO = tmem + TM_O;
            int s = 0;
            uint32_t ph = 0, g = 0;
            bool ok = true;
            for (int qi = 0; ok; ++qi) {
                const int slot = qi & 1;
                if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                if (!INFO(slot)[I_WORK]) break;
                const int nkv = INFO(slot)[I_NKV];
                for (int j = 0; j < nkv; ++j, ++g) {
                    const int pb = int(g & 1u);
                    if (!(ok = bwait(BAR(B_VFULL + s), ph, abort_flag, err))) break;
                    if (!(ok = bwait(BAR(B_PFULL + pb), (g >> 1) & 1u, abort_flag, err))) break;
                    // The item's first product overwrites O: the softmax has read the last one's.
                    if (j == 0 && qi > 0 && !(ok = bwait(BAR(B_OFREE), (qi - 1) & 1, abort_flag, err))) break;
                    tc_fence_after();
                    const uint32_t aP = tmem + TM_P + uint32_t(pb * (BN / 2));
                    const uint64_t dv = dV0 + uint64_t(s * (TILE >> 4));
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        umma_bf16_ts(tO, aP + uint32_t(8 * kk), dv + uint64_t(kk * (2048 >> 4)), idPV,
                                     (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(BAR(B_OFULL + pb));
                    tc_commit(BAR(B_VEMPTY + s));
                    if (++s == NST) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mbar_arrive(BAR(B_IEMPTY + slot));
            }
            tc_commit(BAR(B_FINAL));
            for (int spin = 0; spin < (1 << 24); ++spin)
                if (mbar_try_wait(BAR(B_FINAL), 0)) break;
        }
    } else if (warp < 8) {
        // ------------------------------------------------ softmax (warps 0..7)
        const int half = lane >> 4;
        const int rbase = 32 * (warp & 3) + 16 * (warp >> 2);
        const int r = rbase + (lane & 15);
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tO = tmem + lane_off + TM_O;
        const float c = p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        const SoftmaxWarpB sw{tmem, lane_off, tO, sb + SM_BAR, c2, c, abort_flag, err};
        uint32_t g = 0;
        bool ok = true;
        for (int qi = 0; ok; ++qi) {
            ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_IFULL + (qi & 1)), (qi >> 1) & 1, abort_flag, err));
            if (!ok) break;
            if (!__shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_WORK], 0)) break;
            const int seg_s = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_SEGS], 0);
            const int seg_e = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_SEGE], 0);
            const int nkv = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_NKV], 0);
            float m_ref = 0.0f;
            float l = 0.0f;
            for (int j = 0; j < nkv; ++j, ++g) {
                ok = softmax_tile_bf16(sw, g, seg_s + j * BN + half * HALF, seg_e, j == 0, m_ref, l);
                if (!ok) break;
            }
            if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL + int((g - 1u) & 1u)), ((g - 1u) >> 1) & 1u,
                                                       abort_flag, err));
            if (!ok) break;
            tc_fence_after();
            const int h = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_H], 0);
            const int qrow = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_Q0], 0) + r;
            const bool row_valid = qrow < seg_e;
            const float oscale = 1.0f / (l + __shfl_xor_sync(0xFFFFFFFFu, l, 16));
            uint16_t* orow = p.out + (int64_t(qrow) * p.H + h) * p.D;
            for (int cc = 0; cc < OSPLIT; cc += 16) {
                uint32_t o[16];
                tmem_ld_16x2_x16<OSPLIT>(tO + uint32_t(cc), o);
                tmem_ld_wait16(o);
                uint32_t pkd[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    pkd[q] = cvt_bf16x2(__uint_as_float(o[2 * q]) * oscale, __uint_as_float(o[2 * q + 1]) * oscale);
                const int d0 = half * OSPLIT + cc;
                if (row_valid) {
                    [[maybe_unused]] const int64_t o0 = (int64_t(qrow) * p.H + h) * p.D + d0;   // checked build
                    if (d0 + 8 <= p.D && VF_IN(o0, 8, p.out_elems, err))
                        *reinterpret_cast<uint4*>(orow + d0) = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
                    if (d0 + 16 <= p.D && VF_IN(o0 + 8, 8, p.out_elems, err))
                        *reinterpret_cast<uint4*>(orow + d0 + 8) = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
                }
            }
            // O has been read: the next item's first P.V may overwrite it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(BAR(B_OFREE));
                mbar_arrive(BAR(B_IEMPTY + (qi & 1)));
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

// cuTensorMapEncodeTiled from the driver, looked up once per process
// (thread-safe static initialisation); null if unavailable.
EncodeFnB get_encode_fn_b() {
    static const EncodeFnB fn = []() -> EncodeFnB {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeFnB>(ptr);
        return nullptr;
    }();
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

// Dynamic shared memory opt-in, once per device (a per-device attribute).
PerDeviceOnce g_smem_attr_b;
}  // namespace

vitfp8_status launch_attn_bf16(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* cu, int nseq, int max_seqlen, int T, int H, int D,
                               float sm_scale, uint16_t* out, void* ws, cudaStream_t s) {
    using namespace fb;
    CUtensorMap mq, mk, mv;
    if (!make_map_bf16(&mq, q, T, H, D) || !make_map_bf16(&mk, k, T, H, D) ||
        !make_map_bf16(&mv, v, T, H, D))
        return VITFP8_ERR_CUDA;
    if (launch_attn_plan(cu, nseq, T, H, ROWS_PER_ITEM, 0, 0, ws, s) != cudaSuccess) return VITFP8_ERR_CUDA;
    int dev = -1, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return VITFP8_ERR_CUDA;
    if (!g_smem_attr_b.run(dev, [] {
            return cudaFuncSetAttribute(attn_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_bf16_persistent_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess;
        }))
        return VITFP8_ERR_CUDA;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    AttnParams prm;
    prm.cu = cu;
    prm.rec = reinterpret_cast<const SegRec*>(hdr + 1);
    prm.ws = hdr;
    prm.st = nullptr;
    prm.out = out;
    prm.split_cnt = nullptr;   // no key-range split in this kernel
    prm.split_part = nullptr;
    prm.nseq = nseq;
    prm.T = T;
    prm.H = H;
    prm.D = D;
    prm.Dp = D;
    prm.DV = (D + 15) & ~15;
    prm.KS = (D + 15) / 16;
    prm.sm_scale = sm_scale;
    prm.out_elems = int64_t(T) * H * D;
    const long long grid = (long long)((T + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM + nseq) * H;
    if (grid > 0x7FFFFFFFLL) return VITFP8_ERR_UNSUPPORTED;
    // As for the FP8 path: the persistent kernel for segments of up to 6144
    // tokens when the work items fill more than one wave.
    if (max_seqlen <= 6144 && grid > nsm)
        attn_bf16_persistent_kernel<<<unsigned(nsm), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    else
        attn_bf16_kernel<<<unsigned(grid), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    return cudaGetLastError() == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

}  // namespace vitfp8
