// FP8 variable-length attention, two query tiles per CTA.
//
// "FP8 ViT Encoder Attention", intro and Performance (the FP8 attention
// kernel at head_dim 128; encoder layers at HD / QHD / 4K); "FP8 vision
// encoder attention" (Sonar), Requirements (packed variable-length batches,
// per-tensor scales).  Same arithmetic as attn_fp8.cu (E4M3 scores on the
// tensor cores, online softmax in log2 units against an integer reference,
// P' = E4M3(2^(x - m_ref + 8)), l from a ones block appended to V^T), with a
// different decomposition:
//
//   A work unit is 256 consecutive queries of one (segment, head): query tiles
//   A (rows 0..127) and B (rows 128..255), against every 128-key tile of the
//   segment.  Each softmax thread owns one query row (TMEM access shape
//   32x32b; the row's 128 scores and their maximum come in one load): warps
//   0-3 rows of tile A, warps 4-7 rows of tile B, so every scheduler holds
//   one warp of each tile.  The K and V tiles a unit loads serve 256
//   queries, and a segment has half as many units as 128-row items.
//
//   Up to d = 128 the two tiles share one 128-column S buffer in TMEM:
//   S_A(j), S_B(j), S_A(j+1), ... each wait for the other tile's softmax to
//   have read the buffer, which keeps the A and B warps of a scheduler about
//   half a key tile apart (while one computes exponentials the other loads
//   scores, stores P and rescales O).  For d <= 80 the TMEM columns allow one
//   S buffer per tile, and each tile's next scores are computed while its
//   softmax works on the current ones.
//
//   warp 8      TMA: Q_A and Q_B, then K tiles (128 keys x 128 bytes) and
//               V^T tiles (d rows x 128 keys) through a 4-stage ring.
//   warp 9      S issuer (one thread): S_X(j) = Q_X K_j^T, 128 x 128 per tile.
//   warp 10     P.V issuer (one thread): O_X += P_X(j) V_j, alternating A, B.
//   warp 11     idle (completes the producer warpgroup of the register split).
//
// TMEM columns (512): shared S: S 0..127, O_A 128..271, O_B 272..415, P_A
// 416..447, P_B 448..479 (O holds d + 16 columns: the values and copies of l).
// One S per tile (d <= 80): S_A 0..127, S_B 128..255, O_A 256..351, O_B
// 352..447, P_A 448..479, P_B 480..511.
//
// The reference of a row moves at 128-key instead of 256-key boundaries, so
// its trajectory can differ from attn_fp8.cu's; every reference is a power of
// two, so P' and O differ only where a weight falls in E4M3's subnormal range
// or the fp32 rounding of the exponent argument lands differently (about 1 %
// of outputs by one bf16 ulp on the pages' workloads).
//
// Two kernels run the units: attn_fp8_2tile_kernel one unit per CTA,
// attn_fp8_2tile_persistent_kernel one CTA per SM taking units from a counter
// (for segments of up to 6144 tokens, where a unit's fixed cost weighs most);
// both compute every unit the same way, so their outputs are bit-identical.
//
// Every wait is bounded; on expiry the CTA records VITFP8_ERR_DEVICE_TIMEOUT
// in the workspace error word, all roles leave their loops, wait (bounded)
// for their own async work, free TMEM and return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "host_once.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {
namespace tt {

template <int N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int ID, int COUNT>
__device__ __forceinline__ void named_bar_arrive() {
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}
template <int ID, int COUNT>
__device__ __forceinline__ void named_bar_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

constexpr int BM = 128;                  // rows per query tile
constexpr int BN = 128;                  // keys per key tile
constexpr int NST = 4;                   // K/V ring stages
constexpr int NUM_THREADS = 384;
// setmaxnreg split: 8 softmax warps x 176 + 4 producer warps x 152 registers
// = 64 512, the launch's 384 threads x 168.
constexpr int REGS_SOFTMAX = 176;
constexpr int REGS_PRODUCER = 152;
static_assert(8 * 32 * REGS_SOFTMAX + 4 * 32 * REGS_PRODUCER <= NUM_THREADS * 168, "register split");
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_PV = 10;
constexpr int QBYTES = BM * 128;         // Q tile: 128 rows x 128 bytes
constexpr int KBYTES = BN * 128;         // K tile: 128 keys x 128 bytes
constexpr int VBLK = 144 * 128;          // V^T tile: up to 128 d-rows + 16 rows of ones, x 128 keys
constexpr float PSHIFT = 8.0f;           // P' = 2^(x - m_ref + 8)
constexpr float SLACK = 0.8f;            // x may exceed m_ref by this: P' <= 2^8.8 < 448

constexpr int SM_Q = 0;                  // Q_A, then Q_B
constexpr int SM_K = SM_Q + 2 * QBYTES;
constexpr int SM_V = SM_K + NST * KBYTES;
constexpr int SM_BAR = SM_V + NST * VBLK;

constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_VFULL = B_KFULL + NST;
constexpr int B_KEMPTY = B_VFULL + NST;    // [NST]: S_B of the stage's K tile complete
constexpr int B_VEMPTY = B_KEMPTY + NST;   // [NST]: P_B.V of the stage's V tile complete
constexpr int B_SFULL = B_VEMPTY + NST;    // [2]: S of tile A / B complete
constexpr int B_SFREE = B_SFULL + 2;       // [2]: that S read by the tile's 4 softmax warps
constexpr int B_PFULL = B_SFREE + 2;       // [2]: P written by the tile's 4 softmax warps
constexpr int B_OFULL = B_PFULL + 2;       // [2]: the tile's P.V (and every earlier one) complete
constexpr int B_FINAL = B_OFULL + 2;
// Persistent kernel only:
constexpr int B_QEMPTY = B_FINAL + 1;      // every S product of the current unit is done with Q
constexpr int B_OFREE = B_QEMPTY + 1;      // [2]: the tile's 4 softmax warps have read the unit's O
constexpr int B_IFULL = B_OFREE + 2;       // [2]: unit description written
constexpr int B_IEMPTY = B_IFULL + 2;      // [2]: description used up by all 10 consumers
constexpr int NBAR = B_IEMPTY + 2;
constexpr int IEMPTY_COUNT = 10;           // S issuer, P.V issuer, 8 softmax warps
constexpr int SM_TMEMPTR = SM_BAR + NBAR * 8;
constexpr int SM_ABORT = SM_TMEMPTR + 4;
constexpr int SM_INFO = SM_ABORT + 4;      // persistent: 2 unit descriptions of INFO_INTS ints
constexpr int INFO_INTS = 8;
constexpr int I_WORK = 0, I_H = 1, I_Q0 = 2, I_SEGS = 3, I_SEGE = 4, I_KB0 = 5, I_NKV = 6;
constexpr int SM_USED = SM_INFO + 2 * INFO_INTS * 4;
constexpr int SMEM_BYTES = SM_USED + 1024;  // + slack to align the base to 1024
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;
// Largest O width (d + 16 columns) with one S buffer per tile.
constexpr int OWN_S_MAX_OCOLS = 96;

template <bool OWN_S>
__device__ __forceinline__ uint32_t tm_s(int g) { return OWN_S ? uint32_t(g) * 128u : 0u; }
template <bool OWN_S>
__device__ __forceinline__ uint32_t tm_o(int g) { return OWN_S ? (g ? 352u : 256u) : (g ? 272u : 128u); }
template <bool OWN_S>
__device__ __forceinline__ uint32_t tm_p(int g) { return OWN_S ? (g ? 480u : 448u) : (g ? 448u : 416u); }

template <int N>
__device__ __forceinline__ void scale_words(uint32_t (&o)[N], uint64_t s2) {
#pragma unroll
    for (int q = 0; q < N; q += 2) {
        float a0, a1;
        f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(o[q]), __uint_as_float(o[q + 1])), s2), a0, a1);
        o[q] = __float_as_uint(a0);
        o[q + 1] = __float_as_uint(a1);
    }
}

// O's first nc columns (nc a multiple of 16, <= 144) of this thread's row
// times s (an exact power of two).
__device__ __forceinline__ void rescale_o(uint32_t tO, int nc, float s) {
    const uint64_t s2 = f32x2_pack(s, s);
    int c = 0;
    for (; c + 64 <= nc; c += 64) {
        uint32_t o[64];
        tmem_ld32_x64(tO + uint32_t(c), o);
        scale_words(o, s2);
        tmem_st32_x64_sync(tO + uint32_t(c), o);
    }
    if (c + 32 <= nc) {
        uint32_t o[32];
        tmem_ld32_x32(tO + uint32_t(c), o);
        scale_words(o, s2);
        tmem_st32_x32_sync(tO + uint32_t(c), o);
        c += 32;
    }
    if (c + 16 <= nc) {
        uint32_t o[16];
        tmem_ld32_x16(tO + uint32_t(c), o);
        scale_words(o, s2);
        tmem_st32_x16_sync(tO + uint32_t(c), o);
    }
}

// Softmax of one key tile by one warp of query tile x.g (one thread per row),
// shared by both kernels: wait for the scores, read them with their maximum,
// mask keys outside the segment (first and last tile only), move the row's
// reference when the tile's maximum passes it, wait for the tile's previous
// P.V, write P' = E4M3(2^(x - m_ref + 8)), rescale O and l by the exact power
// of two when the reference moved, and hand P to the P.V issuer.  par is the
// key tile's barrier parity; first marks a unit's first tile (whose P.V wait
// the previous unit's epilogue already did).  False when a wait gave up.
struct Tile2 {
    uint32_t tS, tO, tP;      // this warp's TMEM lanes of S, O and P
    uint32_t bar0;            // shared-memory address of barrier 0
    uint64_t c2;              // (c, c)
    float c;                  // log2 units per raw score
    int nco;                  // O columns: d + 16
    int g;                    // query tile: 0 = A, 1 = B
    volatile int* abort_flag;
    int32_t* err;
};

__device__ __forceinline__ bool softmax_tile2(const Tile2& x, int key0, int seg_s, int seg_e, bool first,
                                              uint32_t par, float& m_ref) {
    const int lane = threadIdx.x & 31;
    auto BAR = [&](int i) -> uint32_t { return x.bar0 + 8u * uint32_t(i); };
    if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_SFULL + x.g), par, x.abort_flag, x.err))) return false;
    tc_fence_after();
    // 128 scores of this row and their maximum.
    float sf[128];
    float pmax;
    tmem_ld32_x128_max(x.tS, sf, pmax);
    // S is in registers: the tensor core may overwrite it.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_SFREE + x.g));

    if (key0 < seg_s || key0 + BN > seg_e) {
        // First or last tile: keys outside the segment are masked and
        // the maximum is taken over the keys left.
#pragma unroll
        for (int i = 0; i < 128; ++i) {
            const int key = key0 + i;
            if ((key < seg_s || key >= seg_e) && VF_IN(i, 1, 128, x.err)) sf[i] = -INFINITY;
        }
        float mx0 = fmaxf(sf[0], sf[1]), mx1 = fmaxf(sf[2], sf[3]);
        float mx2 = fmaxf(sf[4], sf[5]), mx3 = fmaxf(sf[6], sf[7]);
#pragma unroll
        for (int i = 8; i < 128; i += 8) {
            mx0 = fmax3(mx0, sf[i], sf[i + 1]);
            mx1 = fmax3(mx1, sf[i + 2], sf[i + 3]);
            mx2 = fmax3(mx2, sf[i + 4], sf[i + 5]);
            mx3 = fmax3(mx3, sf[i + 6], sf[i + 7]);
        }
        pmax = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
    }
    // Move the reference only when the tile's maximum passes it by
    // more than SLACK; then O and l are rescaled by an exact power of two.
    const float xmax = pmax * x.c;
    float oscale = 1.0f;
    bool need = false;
    if (first) {
        m_ref = ceilf(xmax);
    } else if (xmax > m_ref + SLACK) {
        const float mnew = ceilf(xmax);
        oscale = exp2_int(m_ref - mnew);
        m_ref = mnew;
        need = true;
    }
    if (!first) {
        // The tile's previous P.V is complete (P's columns are free, O
        // with l is final up to that key tile).  Waited for before the
        // exponentials: that product was issued a whole tile ago, and
        // the P store then follows the exponentials without a wait.
        if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL + x.g), par ^ 1u, x.abort_flag, x.err))) return false;
        tc_fence_after();
    }
    const float bias = PSHIFT - m_ref;
    const uint64_t b2 = f32x2_pack(bias, bias);
    // P' = E4M3(2^(x - m_ref + 8)), four keys per 32-bit word.
    uint32_t pk[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        float y0, y1, y2, y3;
        f32x2_unpack(ffma2(f32x2_pack(sf[4 * q], sf[4 * q + 1]), x.c2, b2), y0, y1);
        f32x2_unpack(ffma2(f32x2_pack(sf[4 * q + 2], sf[4 * q + 3]), x.c2, b2), y2, y3);
        pk[q] = cvt_e4m3x4(ex2_approx(y0), ex2_approx(y1), ex2_approx(y2), ex2_approx(y3));
    }
    tmem_st32_x32_sync(x.tP, pk);
    if (__any_sync(0xFFFFFFFFu, need)) rescale_o(x.tO, x.nco, oscale);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_PFULL + x.g));
    return true;
}

// Epilogue of one query row (its thread): o = O * scale_v / l (l = O's column
// DV), rounded to bf16, 16 columns at a time; stored only for rows inside the
// segment.  row0 is the row's first output element.
__device__ __forceinline__ void store_row2(uint32_t tO, const AttnParams& p, float scale_v, int64_t row0,
                                           bool row_valid, int32_t* err) {
    [[maybe_unused]] int32_t* e = err;   // checked build only
    const float l = __uint_as_float(tmem_ld32_x1(tO + uint32_t(p.DV)));
    const float os = scale_v / l;
    uint16_t* orow = p.out + row0;
    for (int c0 = 0; c0 < p.DV; c0 += 16) {
        uint32_t o[16];
        tmem_ld32_x16(tO + uint32_t(c0), o);
        if (!row_valid) continue;
#pragma unroll
        for (int q = 0; q < 16; q += 8) {
            if (c0 + q + 8 > p.D || !VF_IN(row0 + c0 + q, 8, p.out_elems, e)) continue;
            uint4 v;
            v.x = cvt_bf16x2(__uint_as_float(o[q]) * os, __uint_as_float(o[q + 1]) * os);
            v.y = cvt_bf16x2(__uint_as_float(o[q + 2]) * os, __uint_as_float(o[q + 3]) * os);
            v.z = cvt_bf16x2(__uint_as_float(o[q + 4]) * os, __uint_as_float(o[q + 5]) * os);
            v.w = cvt_bf16x2(__uint_as_float(o[q + 6]) * os, __uint_as_float(o[q + 7]) * os);
            *reinterpret_cast<uint4*>(orow + c0 + q) = v;
        }
    }
}

template <bool OWN_S>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_fp8_2tile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    // ---- CTA -> work unit (one record of the work list, 256 rows per unit)
    const int item = blockIdx.x;
    const int4 mine = find_item_load(p);
    const int total = p.ws->total_items;
    SegRec rec;
    if (item >= total || !find_item_pick(p, item, mine, rec)) return;
    const int local = item - rec.first_item;
    const int seg_s = rec.seg_s;
    const int seg_e = rec.seg_e;
    const int nq = rec.nq;
    const int h = local / nq;
    const int qt = local - h * nq;
    const int q0 = seg_s + qt * (2 * BM);
    // Keys are walked from floor16(segment start) so that every V^T copy
    // starts at a 16-byte-aligned token; keys outside the segment are masked.
    const int kb0 = seg_s & ~15;
    const int nkv = (seg_e - kb0 + BN - 1) / BN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM_ABORT);
    int32_t* err = &p.ws->error;
    auto BAR = [&](int i) -> uint32_t { return sb + SM_BAR + 8u * uint32_t(i); };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t vbytes = uint32_t(p.DV) * 128u;

    auto load_k = [&](int j) {
        const int s = j % NST;
        mbar_arrive_expect_tx(BAR(B_KFULL + s), KBYTES);
        tma_load_3d(sb + SM_K + s * KBYTES, &tmK, BAR(B_KFULL + s), 0, h, kb0 + j * BN);
    };
    auto load_v = [&](int j) {
        const int s = j % NST;
        mbar_arrive_expect_tx(BAR(B_VFULL + s), vbytes);
        tma_load_3d(sb + SM_V + s * VBLK, &tmV, BAR(B_VFULL + s), kb0 + j * BN, 0, h);
    };
    // The TMA thread initialises the barriers and starts Q_A, Q_B and K tile
    // 0 before the CTA-wide set-up sync, so they are in flight while the
    // other warps write the ones rows and allocate TMEM.
    if (warp == WARP_TMA && lane == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_KEMPTY + s), 1);
            mbar_init(BAR(B_VEMPTY + s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(BAR(B_SFULL + g), 1);
            mbar_init(BAR(B_SFREE + g), 4);
            mbar_init(BAR(B_PFULL + g), 4);
            mbar_init(BAR(B_OFULL + g), 1);
        }
        mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        // Rows past the tensor's last token arrive as zeros (TMA fill).
        mbar_arrive_expect_tx(BAR(B_QFULL), 2 * QBYTES);
        tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, h, q0);
        tma_load_3d(sb + SM_Q + QBYTES, &tmQ, BAR(B_QFULL), 0, h, q0 + BM);
        if (VF_CHECKED_BUILD && (kb0 & 15) != 0) {
            record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
            *abort_flag = 1;
        } else {
            load_k(0);
        }
    }

    uint32_t tmem = 0;
    if (warp == WARP_TMA) {
        __syncwarp();
        __threadfence_block();
        named_bar_arrive<1, NUM_THREADS>();
    } else {
        // Rows DV..DV+15 of every V^T stage hold E4M3 1.0 (0x38) for good: the
        // TMA boxes cover rows 0..DV-1 only.
        const int t = threadIdx.x < 32 * WARP_TMA ? threadIdx.x : threadIdx.x - 32;
        for (int i = t; i < NST * 16 * 32; i += NUM_THREADS - 32) {
            const int blk = i / (16 * 32);
            const int w = i - blk * (16 * 32);
            if (VF_IN(blk * VBLK + p.DV * 128 + 4 * w, 4, NST * VBLK, err))
                reinterpret_cast<uint32_t*>(smem + SM_V + blk * VBLK + p.DV * 128)[w] = 0x38383838u;
        }
        fence_proxy_async_smem();
        if (warp == WARP_MMA) {
            tmem_alloc(sb + SM_TMEMPTR, TMEM_COLS);
            tmem_relinquish();
        }
        tc_fence_before();
        named_bar_sync<1, NUM_THREADS>();
        tc_fence_after();
        tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEMPTR);
    }

    if (warp >= 8) {
        regs_decrease<REGS_PRODUCER>();
        if (warp == WARP_TMA) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                int issued = 0;   // K/V tiles whose copies were started
                if (!*abort_flag) {
                    load_v(0);
                    issued = 1;
                    for (int j = 1; j < nkv; ++j) {
                        const int s = j % NST;
                        if (j >= NST && !bwait(BAR(B_KEMPTY + s), ((j / NST) - 1) & 1, abort_flag, err)) break;
                        if (j >= NST && !bwait(BAR(B_VEMPTY + s), ((j / NST) - 1) & 1, abort_flag, err)) break;
                        load_k(j);
                        load_v(j);
                        issued = j + 1;
                    }
                }
                if (*abort_flag) {
                    // Let the copies this thread started land before the CTA
                    // exits (bounded spins; these barriers were armed).
                    for (int spin = 0; spin < (1 << 22); ++spin)
                        if (mbar_try_wait(BAR(B_QFULL), 0)) break;
                    for (int jj = (issued > NST ? issued - NST : 0); jj < issued; ++jj) {
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
                const uint32_t idS = make_idesc(0, BM, BN);
                const uint64_t dQA = sw128_kmajor_desc(sb + SM_Q);
                const uint64_t dQB = sw128_kmajor_desc(sb + SM_Q + QBYTES);
                const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
                const int KS = p.KS;
                auto issue_S = [&](uint64_t dQ, int s, int g) {
                    const uint32_t tS = tmem + tm_s<OWN_S>(g);
                    const uint64_t dk = dK0 + uint64_t(s * (KBYTES >> 4));
                    if (KS == 4) {
                        umma_f8_ss_k4(tS, dQ, dk, idS, 0u);
                    } else {
                        umma_f8(tS, dQ, dk, idS, 0u);
                        for (int kk = 1; kk < KS; ++kk)
                            umma_f8(tS, dQ + uint64_t(2 * kk), dk + uint64_t(2 * kk), idS, 1u);
                    }
                };
                bool ok = bwait(BAR(B_QFULL), 0, abort_flag, err);
                for (int j = 0; ok && j < nkv; ++j) {
                    const int s = j % NST;
                    if (!(ok = bwait(BAR(B_KFULL + s), (j / NST) & 1, abort_flag, err))) break;
                    if (OWN_S) {
                        // Each tile's S(j) waits for its own softmax to have read S(j-1).
                        if (j > 0 && !(ok = bwait(BAR(B_SFREE + 0), (j - 1) & 1, abort_flag, err))) break;
                        tc_fence_after();
                        issue_S(dQA, s, 0);
                        tc_commit(BAR(B_SFULL + 0));
                        if (j > 0 && !(ok = bwait(BAR(B_SFREE + 1), (j - 1) & 1, abort_flag, err))) break;
                        tc_fence_after();
                        issue_S(dQB, s, 1);
                    } else {
                        // One buffer: S_A(j) after tile B read S_B(j-1), S_B(j)
                        // after tile A read S_A(j).
                        if (j > 0 && !(ok = bwait(BAR(B_SFREE + 1), (j - 1) & 1, abort_flag, err))) break;
                        tc_fence_after();
                        issue_S(dQA, s, 0);
                        tc_commit(BAR(B_SFULL + 0));
                        if (!(ok = bwait(BAR(B_SFREE + 0), j & 1, abort_flag, err))) break;
                        tc_fence_after();
                        issue_S(dQB, s, 1);
                    }
                    tc_commit(BAR(B_SFULL + 1));
                    tc_commit(BAR(B_KEMPTY + s));
                }
                // Every MMA issued above has completed before TMEM is released.
                tc_commit(BAR(B_FINAL));
                for (int spin = 0; spin < (1 << 24); ++spin)
                    if (mbar_try_wait(BAR(B_FINAL), 0)) break;
            }
        } else if (warp == WARP_PV) {
            // ------------------------------------------------ P.V issuer
            if (lane == 0) {
                const uint32_t idPV = make_idesc(0, BM, p.DV + 16);   // d columns + the l column block
                const uint64_t dV0 = sw128_kmajor_desc(sb + SM_V);
                bool ok = true;
                for (int j = 0; ok && j < nkv; ++j) {
                    // O_X += P_X(j) V_j: 128 keys in 4 steps of 32 (P columns 8 apart).
                    const int s = j % NST;
                    if (!(ok = bwait(BAR(B_VFULL + s), (j / NST) & 1, abort_flag, err))) break;
                    const uint64_t dv = dV0 + uint64_t(s * (VBLK >> 4));
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        if (!(ok = bwait(BAR(B_PFULL + g), j & 1, abort_flag, err))) break;
                        tc_fence_after();
                        umma_f8_ts_k4(tmem + tm_o<OWN_S>(g), tmem + tm_p<OWN_S>(g), dv, idPV, j > 0 ? 1u : 0u);
                        tc_commit(BAR(B_OFULL + g));
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_VEMPTY + s));
                }
                tc_commit(BAR(B_FINAL));
                for (int spin = 0; spin < (1 << 24); ++spin)
                    if (mbar_try_wait(BAR(B_FINAL), 0)) break;
            }
        }
    } else {
        // ------------------------------------------------ softmax (warps 0..7)
        regs_increase<REGS_SOFTMAX>();
        const int g = warp >> 2;                  // query tile: 0 = A, 1 = B
        const int rbase = 32 * (warp & 3);
        const int qrow = q0 + g * BM + rbase + lane;   // packed token index of this row
        const bool row_valid = qrow < seg_e;
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tS = tmem + lane_off + tm_s<OWN_S>(g);
        const uint32_t tO = tmem + lane_off + tm_o<OWN_S>(g);
        const uint32_t tP = tmem + lane_off + tm_p<OWN_S>(g);
        const float c = p.st->scale[0] * p.st->scale[1] * p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        const float scale_v = p.st->scale[2];   // read now: the epilogue needs it last
        const int nco = p.DV + 16;
        float m_ref = 0.0f;
        bool ok = true;
        const Tile2 tx{tS, tO, tP, sb + SM_BAR, c2, c, nco, g, abort_flag, err};
        for (int j = 0; j < nkv; ++j) {
            ok = softmax_tile2(tx, kb0 + j * BN, seg_s, seg_e, j == 0, uint32_t(j) & 1u, m_ref);
            if (!ok) break;
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL + g), uint32_t(nkv - 1) & 1u, abort_flag, err));
        if (ok) {
            tc_fence_after();
            store_row2(tO, p, scale_v, (int64_t(qrow) * p.H + h) * p.D, row_valid, err);
        }
    }

    // ---- teardown: all TMEM traffic of this CTA is complete past this barrier.
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// A unit of the persistent kernel: one 256-query item of the work list.
struct Unit2 {
    int h, q0, seg_s, seg_e, kb0, nkv;
};

// Unit (work item) u -> its rows and key tiles (the calling warp finds the
// record: every lane must call).
__device__ __forceinline__ bool decode_unit2(const AttnParams& p, int u, int4 mine, Unit2& w) {
    SegRec rec;
    if (!find_item_pick(p, u, mine, rec)) return false;
    const int local = u - rec.first_item;
    w.h = local / rec.nq;
    w.q0 = rec.seg_s + (local - w.h * rec.nq) * (2 * BM);
    w.seg_s = rec.seg_s;
    w.seg_e = rec.seg_e;
    w.kb0 = rec.seg_s & ~15;
    w.nkv = (rec.seg_e - w.kb0 + BN - 1) / BN;
    return true;
}

// The same units run by one CTA per SM: the TMA warp takes units from the
// call's counter (the first one is blockIdx.x), publishes each in one of two
// description slots and loads its Q tiles once every S product of the previous
// unit is done with Q, and its K/V tiles through the ring while the previous
// unit finishes, so a unit's set-up and first loads overlap the previous
// unit's last tiles.  Ring stages and the per-tile barrier phases count key
// tiles across units; a unit's first P.V (which overwrites O) waits for the
// tile's softmax warps to have read the previous unit's O.  Every unit
// computes what attn_fp8_2tile_kernel computes for it (same bits).
template <bool OWN_S>
__global__ void __launch_bounds__(NUM_THREADS, 1)
attn_fp8_2tile_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                 const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
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
    const uint32_t vbytes = uint32_t(p.DV) * 128u;
    auto publish = [&](int slot, const Unit2& w) {
        volatile int* inf = INFO(slot);
        inf[I_WORK] = 1;
        inf[I_H] = w.h;
        inf[I_Q0] = w.q0;
        inf[I_SEGS] = w.seg_s;
        inf[I_SEGE] = w.seg_e;
        inf[I_KB0] = w.kb0;
        inf[I_NKV] = w.nkv;
    };

    // The TMA warp decodes the CTA's first unit; its lane 0 initialises the
    // barriers, publishes the unit and starts Q_A, Q_B and K tile 0 before
    // the set-up sync.
    int4 mine = make_int4(0, 0, 0, 0);
    int units = 0;
    Unit2 w0;
    bool have0 = false;
    if (warp == WARP_TMA) {
        mine = find_item_load(p);
        units = p.ws->total_items;
        have0 = int(blockIdx.x) < units && decode_unit2(p, blockIdx.x, mine, w0);
        if (lane == 0) {
            mbar_init(BAR(B_QFULL), 1);
            for (int s = 0; s < NST; ++s) {
                mbar_init(BAR(B_KFULL + s), 1);
                mbar_init(BAR(B_VFULL + s), 1);
                mbar_init(BAR(B_KEMPTY + s), 1);
                mbar_init(BAR(B_VEMPTY + s), 1);
            }
            for (int g = 0; g < 2; ++g) {
                mbar_init(BAR(B_SFULL + g), 1);
                mbar_init(BAR(B_SFREE + g), 4);
                mbar_init(BAR(B_PFULL + g), 4);
                mbar_init(BAR(B_OFULL + g), 1);
                mbar_init(BAR(B_OFREE + g), 4);
                mbar_init(BAR(B_IFULL + g), 1);
                mbar_init(BAR(B_IEMPTY + g), IEMPTY_COUNT);
            }
            mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
            mbar_init(BAR(B_QEMPTY), 1);
            *abort_flag = 0;
            fence_mbar_init();
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            if (have0) publish(0, w0);
            else INFO(0)[I_WORK] = 0;
            mbar_arrive(BAR(B_IFULL + 0));
            if (have0 && VF_CHECKED_BUILD && (w0.kb0 & 15) != 0) {
                record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
                *abort_flag = 1;
            } else if (have0) {
                mbar_arrive_expect_tx(BAR(B_QFULL), 2 * QBYTES);
                tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, w0.h, w0.q0);
                tma_load_3d(sb + SM_Q + QBYTES, &tmQ, BAR(B_QFULL), 0, w0.h, w0.q0 + BM);
                mbar_arrive_expect_tx(BAR(B_KFULL + 0), KBYTES);
                tma_load_3d(sb + SM_K, &tmK, BAR(B_KFULL + 0), 0, w0.h, w0.kb0);
            }
        }
    }

    uint32_t tmem = 0;
    if (warp == WARP_TMA) {
        __syncwarp();
        __threadfence_block();
        named_bar_arrive<1, NUM_THREADS>();
    } else {
        const int t = threadIdx.x < 32 * WARP_TMA ? threadIdx.x : threadIdx.x - 32;
        for (int i = t; i < NST * 16 * 32; i += NUM_THREADS - 32) {
            const int blk = i / (16 * 32);
            const int wd = i - blk * (16 * 32);
            if (VF_IN(blk * VBLK + p.DV * 128 + 4 * wd, 4, NST * VBLK, err))
                reinterpret_cast<uint32_t*>(smem + SM_V + blk * VBLK + p.DV * 128)[wd] = 0x38383838u;
        }
        fence_proxy_async_smem();
        if (warp == WARP_MMA) {
            tmem_alloc(sb + SM_TMEMPTR, TMEM_COLS);
            tmem_relinquish();
        }
        tc_fence_before();
        named_bar_sync<1, NUM_THREADS>();
        tc_fence_after();
        tmem = *reinterpret_cast<volatile uint32_t*>(smem + SM_TMEMPTR);
    }

    if (warp >= 8) {
        regs_decrease<REGS_PRODUCER>();
        if (warp == WARP_TMA) {
            // ------------------------------------------------ TMA producer
            int gt = 0;            // key tiles whose K/V copies were started (across units)
            int kq = 0;            // units whose Q copies were started
            bool k_only = false;   // K of tile gt started, its V not
            bool ok = !*abort_flag;
            Unit2 w = w0;
            bool have = have0;
            for (int qi = 0; ok && have; ++qi) {
                if (lane == 0) {
                    const int slot = qi & 1;
                    if (qi > 0) {
                        if (qi >= 2) ok = bwait(BAR(B_IEMPTY + slot), ((qi - 2) >> 1) & 1, abort_flag, err);
                        if (ok) {
                            publish(slot, w);
                            mbar_arrive(BAR(B_IFULL + slot));
                            if (VF_CHECKED_BUILD && (w.kb0 & 15) != 0) {
                                record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
                                *abort_flag = 1;
                                ok = false;
                            } else if ((ok = bwait(BAR(B_QEMPTY), (qi - 1) & 1, abort_flag, err))) {
                                mbar_arrive_expect_tx(BAR(B_QFULL), 2 * QBYTES);
                                tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, w.h, w.q0);
                                tma_load_3d(sb + SM_Q + QBYTES, &tmQ, BAR(B_QFULL), 0, w.h, w.q0 + BM);
                            }
                        }
                    }
                    if (ok) ++kq;
                    for (int j = 0; ok && j < w.nkv; ++j, ++gt) {
                        const int s = gt % NST;
                        const int key0 = w.kb0 + j * BN;
                        if (!(qi == 0 && j == 0)) {   // K tile 0 of the first unit went out at set-up
                            if (gt >= NST && !(ok = bwait(BAR(B_KEMPTY + s), ((gt / NST) - 1) & 1, abort_flag, err)))
                                break;
                            mbar_arrive_expect_tx(BAR(B_KFULL + s), KBYTES);
                            tma_load_3d(sb + SM_K + s * KBYTES, &tmK, BAR(B_KFULL + s), 0, w.h, key0);
                        }
                        if (gt >= NST && !(ok = bwait(BAR(B_VEMPTY + s), ((gt / NST) - 1) & 1, abort_flag, err))) {
                            k_only = true;
                            break;
                        }
                        mbar_arrive_expect_tx(BAR(B_VFULL + s), vbytes);
                        tma_load_3d(sb + SM_V + s * VBLK, &tmV, BAR(B_VFULL + s), key0, 0, w.h);
                    }
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                // The next unit: every lane takes part in the record vote.
                int nu = 0;
                if (lane == 0) nu = int(gridDim.x) + atomicAdd(&p.ws->next_unit, 1);
                nu = __shfl_sync(0xFFFFFFFFu, nu, 0);
                have = nu < units && decode_unit2(p, nu, mine, w);
                if (!have && lane == 0) {
                    // "No more work" in the next slot, once it is free.
                    const int slot = (qi + 1) & 1;
                    if (qi + 1 < 2 || bwait(BAR(B_IEMPTY + slot), ((qi - 1) >> 1) & 1, abort_flag, err)) {
                        INFO(slot)[I_WORK] = 0;
                        mbar_arrive(BAR(B_IFULL + slot));
                    }
                }
            }
            if (lane == 0 && *abort_flag) {
                // Let the copies this thread started land before the CTA
                // exits (bounded spins; these barriers were armed).
                for (int spin = 0; spin < (1 << 22) && kq > 0; ++spin)
                    if (mbar_try_wait(BAR(B_QFULL), (kq - 1) & 1)) break;
                const int gk = gt + (k_only ? 1 : 0);
                for (int gg = (gk > NST ? gk - NST : 0); gg < gk; ++gg) {
                    const int s = gg % NST;
                    const uint32_t ph = (gg / NST) & 1;
                    for (int spin = 0; spin < (1 << 22); ++spin)
                        if (mbar_try_wait(BAR(B_KFULL + s), ph)) break;
                    for (int spin = 0; spin < (1 << 22) && gg < gt; ++spin)
                        if (mbar_try_wait(BAR(B_VFULL + s), ph)) break;
                }
            }
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------ S issuer
            if (lane == 0) {
                const uint32_t idS = make_idesc(0, BM, BN);
                const uint64_t dQA = sw128_kmajor_desc(sb + SM_Q);
                const uint64_t dQB = sw128_kmajor_desc(sb + SM_Q + QBYTES);
                const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
                const int KS = p.KS;
                auto issue_S = [&](uint64_t dQ, int s, int g) {
                    const uint32_t tS = tmem + tm_s<OWN_S>(g);
                    const uint64_t dk = dK0 + uint64_t(s * (KBYTES >> 4));
                    if (KS == 4) {
                        umma_f8_ss_k4(tS, dQ, dk, idS, 0u);
                    } else {
                        umma_f8(tS, dQ, dk, idS, 0u);
                        for (int kk = 1; kk < KS; ++kk)
                            umma_f8(tS, dQ + uint64_t(2 * kk), dk + uint64_t(2 * kk), idS, 1u);
                    }
                };
                // Key tile gt (counted across units) uses ring stage gt % NST
                // in phase (gt / NST) & 1; its S / P / O barriers, parity gt & 1.
                int gt = 0;
                bool ok = true;
                for (int qi = 0; ok; ++qi) {
                    const int slot = qi & 1;
                    if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                    if (!INFO(slot)[I_WORK]) break;
                    const int nkv = INFO(slot)[I_NKV];
                    if (!(ok = bwait(BAR(B_QFULL), qi & 1, abort_flag, err))) break;
                    for (int j = 0; j < nkv; ++j, ++gt) {
                        const int s = gt % NST;
                        const uint32_t par = uint32_t(gt) & 1u;
                        if (!(ok = bwait(BAR(B_KFULL + s), (gt / NST) & 1, abort_flag, err))) break;
                        if (OWN_S) {
                            if (gt > 0 && !(ok = bwait(BAR(B_SFREE + 0), par ^ 1u, abort_flag, err))) break;
                            tc_fence_after();
                            issue_S(dQA, s, 0);
                            tc_commit(BAR(B_SFULL + 0));
                            if (gt > 0 && !(ok = bwait(BAR(B_SFREE + 1), par ^ 1u, abort_flag, err))) break;
                            tc_fence_after();
                            issue_S(dQB, s, 1);
                        } else {
                            if (gt > 0 && !(ok = bwait(BAR(B_SFREE + 1), par ^ 1u, abort_flag, err))) break;
                            tc_fence_after();
                            issue_S(dQA, s, 0);
                            tc_commit(BAR(B_SFULL + 0));
                            if (!(ok = bwait(BAR(B_SFREE + 0), par, abort_flag, err))) break;
                            tc_fence_after();
                            issue_S(dQB, s, 1);
                        }
                        tc_commit(BAR(B_SFULL + 1));
                        tc_commit(BAR(B_KEMPTY + s));
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_QEMPTY));   // every S product of this unit read Q
                    mbar_arrive(BAR(B_IEMPTY + slot));
                }
                tc_commit(BAR(B_FINAL));
                for (int spin = 0; spin < (1 << 24); ++spin)
                    if (mbar_try_wait(BAR(B_FINAL), 0)) break;
            }
        } else if (warp == WARP_PV) {
            // ------------------------------------------------ P.V issuer
            if (lane == 0) {
                const uint32_t idPV = make_idesc(0, BM, p.DV + 16);
                const uint64_t dV0 = sw128_kmajor_desc(sb + SM_V);
                int gt = 0;
                bool ok = true;
                for (int qi = 0; ok; ++qi) {
                    const int slot = qi & 1;
                    if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                    if (!INFO(slot)[I_WORK]) break;
                    const int nkv = INFO(slot)[I_NKV];
                    for (int j = 0; ok && j < nkv; ++j, ++gt) {
                        const int s = gt % NST;
                        if (!(ok = bwait(BAR(B_VFULL + s), (gt / NST) & 1, abort_flag, err))) break;
                        const uint64_t dv = dV0 + uint64_t(s * (VBLK >> 4));
#pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            if (!(ok = bwait(BAR(B_PFULL + g), uint32_t(gt) & 1u, abort_flag, err))) break;
                            // A unit's first product overwrites O: once the tile's
                            // softmax has read the previous unit's O.
                            if (j == 0 && qi > 0 && !(ok = bwait(BAR(B_OFREE + g), (qi - 1) & 1, abort_flag, err)))
                                break;
                            tc_fence_after();
                            umma_f8_ts_k4(tmem + tm_o<OWN_S>(g), tmem + tm_p<OWN_S>(g), dv, idPV, j > 0 ? 1u : 0u);
                            tc_commit(BAR(B_OFULL + g));
                        }
                        if (!ok) break;
                        tc_commit(BAR(B_VEMPTY + s));
                    }
                    if (!ok) break;
                    mbar_arrive(BAR(B_IEMPTY + slot));
                }
                tc_commit(BAR(B_FINAL));
                for (int spin = 0; spin < (1 << 24); ++spin)
                    if (mbar_try_wait(BAR(B_FINAL), 0)) break;
            }
        }
    } else {
        // ------------------------------------------------ softmax (warps 0..7)
        regs_increase<REGS_SOFTMAX>();
        const int g = warp >> 2;
        const int rbase = 32 * (warp & 3);
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tS = tmem + lane_off + tm_s<OWN_S>(g);
        const uint32_t tO = tmem + lane_off + tm_o<OWN_S>(g);
        const uint32_t tP = tmem + lane_off + tm_p<OWN_S>(g);
        const float c = p.st->scale[0] * p.st->scale[1] * p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        const float scale_v = p.st->scale[2];
        const Tile2 tx{tS, tO, tP, sb + SM_BAR, c2, c, p.DV + 16, g, abort_flag, err};
        int gt = 0;
        bool ok = true;
        for (int qi = 0; ok; ++qi) {
            const int slot = qi & 1;
            ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err));
            if (!ok) break;
            // The unit's description, broadcast from lane 0 (warp-uniform values).
            if (!__shfl_sync(0xFFFFFFFFu, INFO(slot)[I_WORK], 0)) break;
            const int h = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_H], 0);
            const int q0 = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_Q0], 0);
            const int seg_s = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_SEGS], 0);
            const int seg_e = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_SEGE], 0);
            const int kb0 = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_KB0], 0);
            const int nkv = __shfl_sync(0xFFFFFFFFu, INFO(slot)[I_NKV], 0);
            float m_ref = 0.0f;
            for (int j = 0; j < nkv; ++j, ++gt) {
                ok = softmax_tile2(tx, kb0 + j * BN, seg_s, seg_e, j == 0, uint32_t(gt) & 1u, m_ref);
                if (!ok) break;
            }
            if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL + g), uint32_t(gt - 1) & 1u, abort_flag, err));
            if (!ok) break;
            tc_fence_after();
            const int qrow = q0 + g * BM + rbase + lane;
            store_row2(tO, p, scale_v, (int64_t(qrow) * p.H + h) * p.D, qrow < seg_e, err);
            // O has been read: the next unit's first P.V may overwrite it.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(BAR(B_OFREE + g));
                mbar_arrive(BAR(B_IEMPTY + slot));
            }
        }
    }

    // ---- teardown: all TMEM traffic of this CTA is complete past this barrier.
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

PerDeviceOnce g_smem_attr;

}  // namespace tt

vitfp8_status launch_attn_fp8_2tile(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                    const AttnParams& prm, int nsm, bool persistent, cudaStream_t s) {
    using namespace tt;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VITFP8_ERR_CUDA;
    if (launch_attn_plan(prm.cu, prm.nseq, prm.T, prm.H, 2 * BM, nsm, 0, prm.ws, s) != cudaSuccess)
        return VITFP8_ERR_CUDA;
    if (!g_smem_attr.run(dev, [] {
            return cudaFuncSetAttribute(attn_fp8_2tile_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_fp8_2tile_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_fp8_2tile_persistent_kernel<false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_fp8_2tile_persistent_kernel<true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess;
        }))
        return VITFP8_ERR_CUDA;
    // Work units are at most (T / 256 + nseq) * H; CTAs without one return at once.
    const long long units = (long long)((prm.T + 2 * BM - 1) / (2 * BM) + prm.nseq) * prm.H;
    if (units > 0x7FFFFFFFLL) return VITFP8_ERR_UNSUPPORTED;
    const bool own_s = prm.DV + 16 <= OWN_S_MAX_OCOLS;
    if (persistent) {
        // One CTA per SM taking units from the counter the plan zeroed.
        const unsigned grid = unsigned(units < nsm ? units : nsm);
        if (own_s)
            attn_fp8_2tile_persistent_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
        else
            attn_fp8_2tile_persistent_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    } else if (own_s) {
        attn_fp8_2tile_kernel<true><<<unsigned(units), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    } else {
        attn_fp8_2tile_kernel<false><<<unsigned(units), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    }
    return cudaGetLastError() == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

}  // namespace vitfp8
