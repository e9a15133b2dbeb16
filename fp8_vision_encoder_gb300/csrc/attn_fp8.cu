// FP8 variable-length non-causal attention on 5th-generation tensor cores.
//
// "FP8 ViT Encoder Attention", intro: Q/K/V are quantized to FP8 before the
// attention call; Performance: the FP8 attention kernel at head_dim 128,
// seq_len 8192.  "FP8 vision encoder attention" (Sonar), Requirements: packed
// variable-length image batches with per-tensor FP8 scales.
//
// A work unit is one query tile of 128 rows (128 consecutive queries of one
// segment and head) against every key tile of 256 keys of that segment (or a
// key-range part of it, below).  Two kernels run the units with the same
// warp roles and the same arithmetic, so their results are bit-identical:
// attn_fp8_kernel runs one unit per CTA; attn_fp8_persistent_kernel runs one
// CTA per SM that takes units from a counter, its TMA warp loading the next
// unit's Q and K/V tiles while the current unit finishes, so a unit's set-up
// and first loads overlap the previous unit's last tiles.  The two-tile
// kernels (attn_fp8_2tile.cu) run 256-query units with the same arithmetic;
// attn_fp8_kernel_for (internal.cuh) picks one of the four kernels for a call
// (this file's for fewer than two waves of 256-query units, or for long
// segments whose last wave of such units would be far from full).  Roles:
//
//   warp 8      TMA producer: the Q tile once, then K tiles (256 keys x 128 d)
//               and V^T tiles (d x 256 keys) through a shared-memory ring
//               (128-byte swizzle).  Its lane 0 also initialises the barriers
//               and starts the Q tile and the first ring's tiles before the
//               CTA-wide set-up sync, so those copies overlap the set-up.
//   warp 9      S issuer (one thread), tcgen05.mma kind::f8f6f4 (E4M3 x E4M3
//               -> F32) into tensor memory: S(j+1) = Q K_{j+1}^T (N = 256) as
//               soon as the softmax has read S(j).
//   warp 10     P.V issuer (one thread): O += P(j) V_j (P read from TMEM) as
//               soon as P(j) is written.  One thread needs about as long to
//               issue an MMA as the tensor core needs to run it; with two
//               issuers the waits of one overlap the other's MMAs.  The two
//               streams write different accumulators, so their order in the
//               tensor pipe does not matter.
//   warp 11     idle (it completes the producer warpgroup of the register
//               split below).
//   warps 0-7   softmax: warp w owns the 16 rows 32(w%4) + 16(w/4) .. +15;
//               two threads of the warp share each row (TMEM access shape
//               16x32bx2), lanes 0-15 taking the keys 0..127 of a tile and
//               lanes 16-31 the keys 128..255, and combine their row maxima
//               with one shuffle.  No warp waits for another inside a tile.
//
// TMEM (512 columns): S in 0..255 (fp32, 256 keys), O in 256..399, P in
// 448..511 (E4M3, four keys per column).  Because P has its own columns, the
// next S can be computed while the softmax works on the current one: in steady
// state the softmax never waits for the tensor core.  A single thread needs
// about as long to issue one MMA as the tensor core needs to run a 128x128x32
// one; the N = 256 S products halve the number of S instructions.
//
// Softmax in log2 units: x = S_raw * c, c = scale_q scale_k sm_scale log2(e).
// Each row keeps an integer reference m_ref = ceil(running max of x) and
// requantizes P' = E4M3(2^(x - m_ref + 8)), so the row maximum lands in
// (128, 448) (no saturation) and small weights keep E4M3's full range.  The
// reference moves only when a tile's maximum exceeds m_ref by more than 0.8
// (P' would pass 2^8.8): then m_ref = ceil(max) and O and l are rescaled by
// the exact power of two 2^(m_old - m_new).  Because every reference is a
// power of two, the rounded significands equal those taken against the final
// reference (only weights in E4M3's subnormal range, below 2^-6 / 2^8.8 of
// the row maximum, can round differently).
// l sums the rounded P' values themselves (the weights applied to V sum to
// one): each V^T tile carries 16 extra rows of E4M3 ones below its d rows, so
// the P.V product also accumulates l = sum_k P'_k into O's column d = DV, in
// fp32 on the tensor core and rescaled with O.  o = O * scale_v / l, rounded to
// bf16.
//
// Keys are walked in tiles starting at floor16(segment start) so that every
// V^T tile starts at a 16-byte-aligned token coordinate; keys outside the
// segment are masked to -inf (only the first and last tile need it).
//
// Key-range split of the last wave: when the work items leave a last wave
// that would keep at most half the SMs busy for a whole item, the plan cuts
// each item of that wave into up to four parts of consecutive key tiles (one
// unit each).  A part runs the same pipeline over its tiles, stores O, l and
// its reference in the workspace, and the part that finishes last combines
// the parts by exact powers of two and writes the rows.
//
// Every wait (mbarrier or shared-memory handshake) is bounded; on expiry the
// CTA records VITFP8_ERR_DEVICE_TIMEOUT in the workspace error word, all roles
// leave their loops, wait (bounded) for their own async work, free TMEM and
// return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "host_once.h"
#include "internal.cuh"
#include "ptx.cuh"

namespace vitfp8 {

// Per-warpgroup register budget (all four warps of a warpgroup execute the
// same instruction): raise the calling warpgroup's per-thread register count
// to N, or lower it to N and return the rest to the CTA's pool.
template <int N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Named CTA barrier `ID` over `COUNT` threads: arrive without waiting, or
// arrive and wait for all COUNT.
template <int ID, int COUNT>
__device__ __forceinline__ void named_bar_arrive() {
    asm volatile("bar.arrive %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}
template <int ID, int COUNT>
__device__ __forceinline__ void named_bar_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(COUNT) : "memory");
}

namespace fa {
constexpr int BM = 128;                  // query rows per CTA
constexpr int ROWS_PER_ITEM = BM;        // queries per work item
constexpr int BN = 256;                  // keys per tile
constexpr int HALF = BN / 2;             // keys per softmax thread and tile
constexpr int NST = 3;                   // K/V pipeline stages
constexpr int NUM_THREADS = 384;         // 8 softmax warps; TMA warp, S and P.V issuers, one idle warp
// Registers: a launch of 384 threads gives every thread 168 (a scheduler hosts
// three of the twelve warps).  Each warpgroup then moves to its own budget at
// the top of its branch: the two softmax warpgroups up to REGS_SOFTMAX (a
// 128-score half row, its 32 P words and the O rescale), the producer
// warpgroup (TMA, the two issuers, an idle warp) down to REGS_PRODUCER.
// 176 against the 160 a uniform budget allows: the compiler then schedules the
// softmax loop with fewer stalls (about 1.5 % per tile on the 3xQHD layer);
// 152 keeps the producer warpgroup free of spills.
constexpr int REGS_SOFTMAX = 176;
constexpr int REGS_PRODUCER = 152;
static_assert(8 * 32 * REGS_SOFTMAX + 4 * 32 * REGS_PRODUCER <= NUM_THREADS * 168, "register split");
// The persistent kernel's producer warpgroup decodes work units and keeps
// their state: 136 registers keep it free of spills, 184 go to the softmax.
constexpr int REGS_SOFTMAX_P = 184;
constexpr int REGS_PRODUCER_P = 136;
static_assert(8 * 32 * REGS_SOFTMAX_P + 4 * 32 * REGS_PRODUCER_P <= NUM_THREADS * 168, "register split");
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;              // S issuer; owns the TMEM allocation
constexpr int WARP_PV = 10;              // P.V issuer
constexpr int QBYTES = BM * 128;         // Q tile: 128 rows x 128 bytes
constexpr int KBYTES = BN * 128;         // K tile: 256 rows x 128 bytes
constexpr int VBLK = 144 * 128;          // V^T block: up to 128 d-rows + 16 rows of ones, x 128 keys
constexpr int VBYTES = 2 * VBLK;         // V^T tile: two key blocks
constexpr float PSHIFT = 8.0f;           // P' = 2^(x - m_ref + 8)
constexpr float SLACK = 0.8f;            // x may exceed m_ref by this: P' <= 2^8.8 < 448

constexpr int SM_Q = 0;
constexpr int SM_K = SM_Q + QBYTES;
constexpr int SM_V = SM_K + NST * KBYTES;
constexpr int SM_BAR = SM_V + NST * VBYTES;
// barrier indices
constexpr int B_QFULL = 0;
constexpr int B_KFULL = 1;
constexpr int B_VFULL = B_KFULL + NST;
constexpr int B_KEMPTY = B_VFULL + NST;    // [NST]: S of the stage's K tile complete
constexpr int B_VEMPTY = B_KEMPTY + NST;   // [NST]: P.V of the stage's V tile complete
constexpr int B_SFULL = B_VEMPTY + NST;    // S(j) complete in TMEM
constexpr int B_SFREE = B_SFULL + 1;       // S(j) read by all 8 softmax warps
constexpr int B_PFULL = B_SFREE + 1;       // P(j) written by all 8 softmax warps
constexpr int B_OFULL = B_PFULL + 1;       // P(j) V_j (and every earlier MMA) complete
constexpr int B_FINAL = B_OFULL + 1;
constexpr int B_QEMPTY = B_FINAL + 1;      // every S product of the current item is done with Q
constexpr int B_OFREE = B_QEMPTY + 1;      // the 8 softmax warps have read the item's O
constexpr int B_IFULL = B_OFREE + 1;       // [2]: work-item description written
constexpr int B_IEMPTY = B_IFULL + 2;      // [2]: description used up by all 10 consumers
constexpr int NBAR = B_IEMPTY + 2;
constexpr int IEMPTY_COUNT = 10;           // S issuer, P.V issuer, 8 softmax warps
constexpr int SM_TMEMPTR = SM_BAR + NBAR * 8;
constexpr int SM_ABORT = SM_TMEMPTR + 4;
constexpr int SM_LAST = SM_ABORT + 4;      // key-range split: this CTA merges the parts
constexpr int SM_SPLIT = SM_LAST + 4;      // one item per CTA: split slot, item index, parts (3 ints)
constexpr int SM_INFO = SM_SPLIT + 12;     // persistent: 2 work-unit descriptions of INFO_INTS ints
constexpr int INFO_INTS = 16;
constexpr int SM_USED = SM_INFO + 2 * INFO_INTS * 4;
// Work-unit description (ints): I_WORK 1 for a unit, 0 for "no more work".
constexpr int I_WORK = 0, I_H = 1, I_Q0 = 2, I_SEGS = 3, I_SEGE = 4, I_KB0 = 5, I_NKV = 6,
              I_SLOT = 7, I_GRP = 8, I_PARTS = 9;
constexpr int SMEM_BYTES = SM_USED + 1024;  // + slack to align the base to 1024
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0, TM_O = 256, TM_P = 448;
constexpr int OSPLIT = 80;               // O columns per half-row thread (2 x 80 >= 128 + 16)
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
// A split part's partial results: per softmax thread its OSPLIT O columns
// (OSPLIT / 4 chunks of four floats, chunk-major so a warp's stores coalesce),
// then (l, m_ref) per thread.
constexpr int PART_CHUNKS = OSPLIT / 4;
constexpr int PART_LM = PART_CHUNKS * 256 * 4;   // float offset of the (l, m_ref) pairs
constexpr int PART_FLOATS = PART_LM + 2 * 256;
static_assert(PART_FLOATS * sizeof(float) <= kSplitPartBytes, "split part fits its slot");
}  // namespace fa

// Epilogue of one part of a split work item (softmax threads 0..255, called
// by all of them): slot = its part's index among the split CTAs, grp = its
// item's index among the split items, sp_k = parts per item.  O, l and the reference cover this part's key tiles only.
// Every part stores them in its workspace slot (output columns < D only); the
// part that arrives last combines all parts in part order, so the result does
// not depend on which part that is:
//   M = max_p m_p,  O = sum_p O_p 2^(m_p - M),  l = sum_p l_p 2^(m_p - M),
// exact powers of two as in the single-pass rescale.  Kept out of line so
// that it does not take registers from the tile loop.
struct SplitOut {
    float* part;          // the workspace's partial-result slots
    int32_t* cnt;         // per split item: parts finished
    uint16_t* out;        // bf16 output row of this thread's query (h included)
    int32_t* err;
    int64_t out_off;      // that row's first element index (checked build)
    int64_t out_elems;
    int D, DV;
};

__device__ __noinline__ void split_part_epilogue(const SplitOut so, uint32_t tO, bool row_valid, int half,
                                                 float m_ref, float scale_v, int slot, int grp, int sp_k,
                                                 bool ok, volatile int* abort_flag, uint8_t* last_flag,
                                                 uint32_t ofree_bar) {
    using namespace fa;
    [[maybe_unused]] int32_t* err = so.err;   // checked build only
    const int tid = threadIdx.x;   // 0..255: the softmax threads
    const int cbase = half * OSPLIT;
    constexpr size_t PSTRIDE = kSplitPartBytes / sizeof(float);
    if (!VF_IN(slot, 1, kSplitMaxParts, err)) ok = false;
    if (ok) {
        tc_fence_after();
        uint32_t lbits;
        uint32_t oa[32], ob[32], oc[16];
        tmem_ld_o80<OSPLIT>(tO, tO + uint32_t(so.DV), oa, ob, oc, lbits);
        float* mine = so.part + size_t(slot) * PSTRIDE;
        uint4* dst = reinterpret_cast<uint4*>(mine);
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
            if (cbase + 4 * q + 8 <= so.D) {
                __stcg(dst + q * 256 + tid, make_uint4(oa[4 * q], oa[4 * q + 1], oa[4 * q + 2], oa[4 * q + 3]));
                __stcg(dst + (q + 1) * 256 + tid,
                       make_uint4(oa[4 * q + 4], oa[4 * q + 5], oa[4 * q + 6], oa[4 * q + 7]));
            }
            if (cbase + 32 + 4 * q + 8 <= so.D) {
                __stcg(dst + (8 + q) * 256 + tid, make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]));
                __stcg(dst + (9 + q) * 256 + tid,
                       make_uint4(ob[4 * q + 4], ob[4 * q + 5], ob[4 * q + 6], ob[4 * q + 7]));
            }
        }
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
            if (cbase + 64 + 4 * q + 8 <= so.D) {
                __stcg(dst + (16 + q) * 256 + tid,
                       make_uint4(oc[4 * q], oc[4 * q + 1], oc[4 * q + 2], oc[4 * q + 3]));
                __stcg(dst + (17 + q) * 256 + tid,
                       make_uint4(oc[4 * q + 4], oc[4 * q + 5], oc[4 * q + 6], oc[4 * q + 7]));
            }
        }
        __stcg(reinterpret_cast<float2*>(mine + PART_LM) + tid, make_float2(__uint_as_float(lbits), m_ref));
    }
    // O has been read: the next unit's first P.V may overwrite it (persistent
    // kernel; 0 when the CTA has no next unit).
    if (ofree_bar != 0u) {
        tc_fence_before();
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(ofree_bar);
    }
    __threadfence();
    named_bar_sync<2, 256>();
    if (tid == 0) {
        int last = 0;
        if (!*abort_flag && VF_IN(grp, 1, kSplitMaxParts, err))
            last = atomicAdd(so.cnt + grp, 1) == sp_k - 1;
        *reinterpret_cast<volatile int*>(last_flag) = last;
    }
    named_bar_sync<2, 256>();
    if (!ok || !*reinterpret_cast<volatile int*>(last_flag)) return;
    __threadfence();
    const float* base = so.part + size_t(grp) * sp_k * PSTRIDE;
    float f[kSplitMaxK], lp[kSplitMaxK];
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kSplitMaxK; ++q) {
        if (q < sp_k) {
            const float2 lm = __ldcg(reinterpret_cast<const float2*>(base + q * PSTRIDE + PART_LM) + tid);
            lp[q] = lm.x;
            f[q] = lm.y;
            M = fmaxf(M, lm.y);
        }
    }
    float l = 0.0f;
#pragma unroll
    for (int q = 0; q < kSplitMaxK; ++q) {
        if (q < sp_k) {
            f[q] = exp2_int(f[q] - M);
            l += lp[q] * f[q];
        }
    }
    const float oscale = scale_v / l;
    uint16_t* orow = so.out;
#pragma unroll 1
    for (int c = 0; c < PART_CHUNKS; c += 2) {
        const int d0 = cbase + 4 * c;
        if (d0 + 8 > so.D) break;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int q = 0; q < kSplitMaxK; ++q) {
            if (q < sp_k) {
                const uint4* src = reinterpret_cast<const uint4*>(base + q * PSTRIDE);
                const uint4 a = __ldcg(src + c * 256 + tid);
                const uint4 b = __ldcg(src + (c + 1) * 256 + tid);
                acc[0] += __uint_as_float(a.x) * f[q];
                acc[1] += __uint_as_float(a.y) * f[q];
                acc[2] += __uint_as_float(a.z) * f[q];
                acc[3] += __uint_as_float(a.w) * f[q];
                acc[4] += __uint_as_float(b.x) * f[q];
                acc[5] += __uint_as_float(b.y) * f[q];
                acc[6] += __uint_as_float(b.z) * f[q];
                acc[7] += __uint_as_float(b.w) * f[q];
            }
        }
        if (!row_valid || !VF_IN(so.out_off + d0, 8, so.out_elems, err)) continue;
        uint4 v;
        v.x = cvt_bf16x2(acc[0] * oscale, acc[1] * oscale);
        v.y = cvt_bf16x2(acc[2] * oscale, acc[3] * oscale);
        v.z = cvt_bf16x2(acc[4] * oscale, acc[5] * oscale);
        v.w = cvt_bf16x2(acc[6] * oscale, acc[7] * oscale);
        *reinterpret_cast<uint4*>(orow + d0) = v;
    }
}

// Softmax of one key tile, shared by both kernels (the 8 softmax warps, two
// threads per row): wait for S, read it with its maximum, mask
// keys outside the segment (first and last tile only), move the row's
// reference when the tile's maximum passes it (O and l rescaled by an exact
// power of two), write P' = E4M3(2^(x - m_ref + 8)) and signal P.V.  gpar is
// the tile's barrier parity; first marks a unit's first tile.  key0 is this
// thread's first key.  False when a wait gave up.
struct SoftmaxWarp {
    uint32_t tS, tO, tP;      // this warp's TMEM lanes of S, O and P
    uint32_t bar0;            // shared-memory address of barrier 0
    uint64_t c2;              // (c, c)
    float c;                  // log2 units per raw score
    int DV;
    volatile int* abort_flag;
    int32_t* err;
};

__device__ __forceinline__ bool softmax_tile(const SoftmaxWarp& x, int key0, int seg_s, int seg_e, bool first,
                                             uint32_t gpar, float& m_ref) {
    using namespace fa;
    const int lane = threadIdx.x & 31;
    auto BAR = [&](int i) -> uint32_t { return x.bar0 + 8u * uint32_t(i); };
    if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_SFULL), gpar, x.abort_flag, x.err))) return false;
    tc_fence_after();
    // One load returns the 128 scores and their maximum (tcgen05.ld.red).
    float sf[128];
    float pmax;
    tmem_ld_s128_max<HALF>(x.tS, sf, pmax);
    // S is in registers: the tensor core may overwrite it with the next S.
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_SFREE));

    if (key0 < seg_s || key0 + HALF > seg_e) {
        // First or last tile: keys outside the segment are masked, and
        // the maximum is taken over the keys left.
#pragma unroll
        for (int i = 0; i < 128; ++i) {
            const int key = key0 + i;
            if ((key < seg_s || key >= seg_e) && VF_IN(i, 1, 128, x.err)) sf[i] = -INFINITY;
        }
        // Four running maxima over sf[0..127]: pairs 0..7 seed them,
        // then eight values per step.
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
    // Row maximum over both key halves (lane ^ 16 holds the other half).
    pmax = fmaxf(pmax, __shfl_xor_sync(0xFFFFFFFFu, pmax, 16));
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

    if (!first) {
        // The previous tile's P.V complete: P's columns are free and O
        // (with l) is final up to that tile (needed before a rescale).
        // Before a unit's first tile there is none (or the previous
        // unit's epilogue waited for it).
        if (!__all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL), gpar ^ 1u, x.abort_flag, x.err))) return false;
        tc_fence_after();
    }
    if (__any_sync(0xFFFFFFFFu, need)) {
        // O's DV + 16 columns (values, then copies of l): lanes 0-15
        // scale columns 0..79, lanes 16-31 columns 80..159 (columns
        // past DV + 16 are unused TMEM).
        const uint64_t s2v = f32x2_pack(oscale, oscale);
        uint32_t oa[32], ob[32], oc[16], lunused;
        tmem_ld_o80<OSPLIT>(x.tO, x.tO + uint32_t(x.DV), oa, ob, oc, lunused);
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
#pragma unroll
        for (int q = 0; q < 16; q += 2) {
            float a0, a1;
            f32x2_unpack(fmul2(f32x2_pack(__uint_as_float(oc[q]), __uint_as_float(oc[q + 1])), s2v), a0, a1);
            oc[q] = __float_as_uint(a0);
            oc[q + 1] = __float_as_uint(a1);
        }
        tmem_st_o80_sync<OSPLIT>(x.tO, oa, ob, oc);
    }
    // This half of the P row: 128 keys in 32 columns (lanes 16-31 at +32).
    tmem_st_16x2_x32_sync<HALF / 4>(x.tP, pk);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_PFULL));
    return true;
}

__global__ void __launch_bounds__(fa::NUM_THREADS, 1)
attn_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace fa;
    // ---- CTA -> work item and key-range part.  Items from split_first on are
    // cut into split_k parts of consecutive key tiles, one CTA each.
    // Every load the decode needs goes out at once: the header (item count
    // and split), and with at most 32 segments each lane's record.
    const int cta = blockIdx.x;
    const int4 mine = find_item_load(p);
    const int4 hdr = *reinterpret_cast<const int4*>(p.ws);   // error, total_items, num_seqs, split_first
    const int split_k = p.ws->split_k;
    const int total = hdr.y;
    const int split_first = hdr.w;
    int item = cta, part = 0, nparts = 1;
    if (split_k > 1 && cta >= split_first) {
        const int d = cta - split_first;
        item = split_first + d / split_k;
        part = d - (d / split_k) * split_k;
        nparts = split_k;
    }
    // ---- work item -> (segment, head, query tile): one record of the work list
    SegRec rec;
    if (item >= total || !find_item_pick(p, item, mine, rec)) return;
    const int local = item - rec.first_item;
    const int seg_s = rec.seg_s;
    const int seg_e = rec.seg_e;
    const int nq = rec.nq;
    const int h = local / nq;
    const int qt = local - h * nq;
    const int q0 = seg_s + qt * ROWS_PER_ITEM;
    const int kbase = seg_s & ~15;
    const int nkv_all = (seg_e - kbase + BN - 1) / BN;
    // This part's key tiles t0 .. t0 + nkv - 1 (all of them when not split;
    // the plan gives every part at least one).
    const int t0 = nkv_all * part / nparts;
    const int nkv = nkv_all * (part + 1) / nparts - t0;
    const int kb0 = kbase + t0 * BN;
    if (VF_CHECKED_BUILD && (nkv < 1 || (nparts > 1 && (item - split_first >= kSplitMaxParts ||
                                                         cta - split_first >= kSplitMaxParts)))) {
        if (threadIdx.x == 0) record_error(&p.ws->error, VITFP8_ERR_DEVICE_BOUNDS);
        return;
    }

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
        // For the epilogue (read after the set-up sync, so that these values
        // do not stay live through the tile loop): split slot, split item, parts.
        int* spl = reinterpret_cast<int*>(smem + SM_SPLIT);
        spl[0] = cta - split_first;
        spl[1] = item - split_first;
        spl[2] = nparts;
    }

    // The TMA thread initialises the barriers and starts the copies the first
    // S product needs (the Q tile and K tile 0) at once, so they are in flight
    // while the CTA sets up the ones rows and TMEM; the rest of the first ring
    // follows right after the CTA-wide sync (no other thread touches a
    // barrier before it).
    const uint32_t vbytes = 2u * uint32_t(p.DV) * 128u;
    auto load_k = [&](int j) {
        const int s = j % NST;
        mbar_arrive_expect_tx(BAR(B_KFULL + s), KBYTES);
        tma_load_3d(sb + SM_K + s * KBYTES, &tmK, BAR(B_KFULL + s), 0, h, kb0 + j * BN);
    };
    auto load_v = [&](int j) {
        const int s = j % NST;
        const int key0 = kb0 + j * BN;
        mbar_arrive_expect_tx(BAR(B_VFULL + s), vbytes);
        tma_load_3d(sb + SM_V + s * VBYTES, &tmV, BAR(B_VFULL + s), key0, 0, h);
        tma_load_3d(sb + SM_V + s * VBYTES + VBLK, &tmV, BAR(B_VFULL + s), key0 + HALF, 0, h);
    };
    if (warp == WARP_TMA && lane == 0) {
        mbar_init(BAR(B_QFULL), 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(BAR(B_KFULL + s), 1);
            mbar_init(BAR(B_VFULL + s), 1);
            mbar_init(BAR(B_KEMPTY + s), 1);
            mbar_init(BAR(B_VEMPTY + s), 1);
        }
        mbar_init(BAR(B_SFULL), 1);
        mbar_init(BAR(B_SFREE), 8);
        mbar_init(BAR(B_PFULL), 8);
        mbar_init(BAR(B_OFULL), 1);
        mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(BAR(B_QFULL), QBYTES);
        tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, h, q0);
        // V^T copies start at token kb0 + j * BN, a multiple of 16: TMA needs
        // the innermost coordinate 16-byte aligned (checked in the checked build).
        if (VF_CHECKED_BUILD && (kb0 & 15) != 0) {
            record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
            *abort_flag = 1;
        } else {
            load_k(0);
        }
    }

    // Set-up sync on named barrier 1: the TMA warp only arrives (once the
    // barriers are initialised) and goes straight on with its copies; every
    // other warp also writes the ones rows and allocates TMEM, then waits.
    uint32_t tmem = 0;
    if (warp == WARP_TMA) {
        __syncwarp();
        __threadfence_block();
        named_bar_arrive<1, NUM_THREADS>();
    } else {
        // Rows DV..DV+15 of every V^T block hold E4M3 1.0 (0x38) for good:
        // the TMA boxes cover rows 0..DV-1 only.  (Uniform bytes: the swizzle
        // does not matter.)  The tensor core reads them through the async
        // proxy.
        const int t = threadIdx.x < 32 * WARP_TMA ? threadIdx.x : threadIdx.x - 32;
        for (int i = t; i < NST * 2 * 16 * 32; i += NUM_THREADS - 32) {
            const int blk = i / (16 * 32);
            const int w = i - blk * (16 * 32);
            if (VF_IN(blk * VBLK + p.DV * 128 + 4 * w, 4, NST * VBYTES, &p.ws->error))
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
                // The Q tile and K tile 0 are in flight since the set-up
                // (neither K nor V if the set-up found kb0 misaligned): V
                // tile 0 and K/V tiles 1..NST-1 go at once, while the other
                // warps finish their set-up; tile j >= NST reuses its stage
                // once S and P.V of tile j - NST are done with it.
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
                const uint32_t idS = make_idesc(0, BM, BN);      // 128 x 256 per S product
                // Descriptors are built once: within a 128-byte swizzled row a
                // 32-byte K step adds 2 to the encoded start address; a stage
                // adds its byte offset / 16.
                const uint64_t dQ = sw128_kmajor_desc(sb + SM_Q);
                const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
                const uint32_t tS = tmem + TM_S;
                const int KS = p.KS;
                auto issue_S = [&](int s) {
                    const uint64_t dk = dK0 + uint64_t(s * (KBYTES >> 4));
                    if (KS == 4) {
                        umma_f8_ss_k4(tS, dQ, dk, idS, 0u);
                    } else {
                        umma_f8(tS, dQ, dk, idS, 0u);
                        for (int kk = 1; kk < KS; ++kk)
                            umma_f8(tS, dQ + uint64_t(2 * kk), dk + uint64_t(2 * kk), idS, 1u);
                    }
                    tc_commit(BAR(B_SFULL));
                    tc_commit(BAR(B_KEMPTY + s));
                };
                bool ok = bwait(BAR(B_QFULL), 0, abort_flag, err) &&
                          bwait(BAR(B_KFULL + 0), 0, abort_flag, err);
                if (ok) {
                    tc_fence_after();
                    issue_S(0);
                }
                int s1 = 1 % NST;
                uint32_t ph1 = NST == 1 ? 1u : 0u;
                for (int j = 0; ok && j + 1 < nkv; ++j) {
                    // S(j+1) as soon as K_{j+1} is in and every softmax warp has read S(j).
                    if (!(ok = bwait(BAR(B_KFULL + s1), ph1, abort_flag, err))) break;
                    if (!(ok = bwait(BAR(B_SFREE), j & 1, abort_flag, err))) break;
                    tc_fence_after();
                    issue_S(s1);
                    if (++s1 == NST) {
                        s1 = 0;
                        ph1 ^= 1u;
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
                const uint32_t idPV = make_idesc(0, BM, p.DV + 16);   // d columns + the l column block
                const uint64_t dV0 = sw128_kmajor_desc(sb + SM_V);
                const uint32_t tO = tmem + TM_O, tP = tmem + TM_P;
                int s = 0;
                uint32_t ph = 0;
                bool ok = true;
                for (int j = 0; ok && j < nkv; ++j) {
                    // O += P(j) V_j: 256 keys in 8 steps of 32, keys 0..127 from
                    // V^T block 0 and P columns 0..31, keys 128..255 from block 1
                    // and P columns 32..63.
                    if (!(ok = bwait(BAR(B_VFULL + s), ph, abort_flag, err))) break;
                    if (!(ok = bwait(BAR(B_PFULL), j & 1, abort_flag, err))) break;
                    tc_fence_after();
                    const uint64_t dv = dV0 + uint64_t(s * (VBYTES >> 4));
                    umma_f8_ts_k4(tO, tP, dv, idPV, j > 0 ? 1u : 0u);
                    umma_f8_ts_k4(tO, tP + 32u, dv + uint64_t(VBLK >> 4), idPV, 1u);
                    tc_commit(BAR(B_OFULL));
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
        }
    } else {
        // ------------------------------------------------ softmax (warps 0..7)
        regs_increase<REGS_SOFTMAX>();
        const int half = lane >> 4;           // keys half*128 .. half*128+127 of each tile
        const int rbase = 32 * (warp & 3) + 16 * (warp >> 2);
        const int r = rbase + (lane & 15);    // row inside the query tile
        const int qrow = q0 + r;              // packed token index of this row
        const bool row_valid = qrow < seg_e;
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tS = tmem + lane_off + TM_S;
        const uint32_t tO = tmem + lane_off + TM_O;
        const uint32_t tP = tmem + lane_off + TM_P;
        const float c = p.st->scale[0] * p.st->scale[1] * p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        const float scale_v = p.st->scale[2];   // read now: the epilogue needs it last
        float m_ref = 0.0f;
        bool ok = true;
        const SoftmaxWarp sw{tS, tO, tP, sb + SM_BAR, c2, c, p.DV, abort_flag, err};
        for (int j = 0; j < nkv; ++j) {
            ok = softmax_tile(sw, kb0 + j * BN + half * HALF, seg_s, seg_e, j == 0, uint32_t(j) & 1u, m_ref);
            if (!ok) break;
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL), (nkv - 1) & 1, abort_flag, err));
        uint16_t* orow = p.out + (int64_t(qrow) * p.H + h) * p.D;
        const int cbase = half * OSPLIT;
        // Eight output columns d0..d0+7 of this row: o = O * oscale, rounded to bf16.
        auto store8 = [&](int d0, float oscale, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                          uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
            if (!row_valid || d0 + 8 > p.D) return;
            if (!VF_IN((int64_t(qrow) * p.H + h) * p.D + d0, 8, p.out_elems, err)) return;
            uint4 v;
            v.x = cvt_bf16x2(__uint_as_float(a0) * oscale, __uint_as_float(a1) * oscale);
            v.y = cvt_bf16x2(__uint_as_float(a2) * oscale, __uint_as_float(a3) * oscale);
            v.z = cvt_bf16x2(__uint_as_float(a4) * oscale, __uint_as_float(a5) * oscale);
            v.w = cvt_bf16x2(__uint_as_float(a6) * oscale, __uint_as_float(a7) * oscale);
            *reinterpret_cast<uint4*>(orow + d0) = v;
        };
        const int* spl = reinterpret_cast<const int*>(smem + SM_SPLIT);
        const int sp_k = spl[2];   // parts of this CTA's work item (1: not split)
        if (sp_k == 1) {
            if (ok) {
                tc_fence_after();
                uint32_t lbits;   // both halves: a copy of l (column DV)
                uint32_t oa[32], ob[32], oc[16];
                tmem_ld_o80<OSPLIT>(tO, tO + uint32_t(p.DV), oa, ob, oc, lbits);
                const float oscale = scale_v / __uint_as_float(lbits);
#pragma unroll
                for (int q = 0; q < 32; q += 8) {
                    store8(cbase + q, oscale, oa[q], oa[q + 1], oa[q + 2], oa[q + 3], oa[q + 4], oa[q + 5],
                           oa[q + 6], oa[q + 7]);
                    store8(cbase + 32 + q, oscale, ob[q], ob[q + 1], ob[q + 2], ob[q + 3], ob[q + 4],
                           ob[q + 5], ob[q + 6], ob[q + 7]);
                }
                store8(cbase + 64, oscale, oc[0], oc[1], oc[2], oc[3], oc[4], oc[5], oc[6], oc[7]);
                store8(cbase + 72, oscale, oc[8], oc[9], oc[10], oc[11], oc[12], oc[13], oc[14], oc[15]);
            }
        } else {
            SplitOut so;
            so.part = p.split_part;
            so.cnt = p.split_cnt;
            so.out = orow;
            so.err = err;
            so.out_off = (int64_t(qrow) * p.H + h) * p.D;
            so.out_elems = p.out_elems;
            so.D = p.D;
            so.DV = p.DV;
            split_part_epilogue(so, tO, row_valid, half, m_ref, scale_v, spl[0], spl[1], sp_k, ok, abort_flag,
                                smem + SM_LAST, 0u);
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

// A work unit: one work item, or one key-range part of a split item.
struct Unit {
    int h, q0, seg_s, seg_e, kb0, nkv;
    int slot, grp, parts;   // split part index, split item index, parts per item (1: not split)
};

// Unit u -> its work item (one record of the work list, found by the calling
// warp: every lane must call) and its key tiles.  Units from split_first on
// are the parts of split items, split_k per item.
__device__ __forceinline__ bool decode_unit(const AttnParams& p, int u, int split_first, int split_k,
                                            int4 mine, Unit& w) {
    using namespace fa;
    int item = u, part = 0, parts = 1;
    if (split_k > 1 && u >= split_first) {
        const int d = u - split_first;
        item = split_first + d / split_k;
        part = d - (d / split_k) * split_k;
        parts = split_k;
    }
    SegRec rec;
    if (!find_item_pick(p, item, mine, rec)) return false;
    const int local = item - rec.first_item;
    const int nq = rec.nq;
    w.h = local / nq;
    w.q0 = rec.seg_s + (local - w.h * nq) * ROWS_PER_ITEM;
    w.seg_s = rec.seg_s;
    w.seg_e = rec.seg_e;
    const int kbase = rec.seg_s & ~15;
    const int nkv_all = (rec.seg_e - kbase + BN - 1) / BN;
    const int t0 = nkv_all * part / parts;
    w.nkv = nkv_all * (part + 1) / parts - t0;
    w.kb0 = kbase + t0 * BN;
    w.slot = u - split_first;
    w.grp = item - split_first;
    w.parts = parts;
    if (VF_CHECKED_BUILD && (w.nkv < 1 || (parts > 1 && (w.slot >= kSplitMaxParts || w.grp >= kSplitMaxParts)))) {
        record_error(&p.ws->error, VITFP8_ERR_DEVICE_BOUNDS);
        return false;
    }
    return true;
}

__global__ void __launch_bounds__(fa::NUM_THREADS, 1)
attn_fp8_persistent_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using namespace fa;
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
    const uint32_t vbytes = 2u * uint32_t(p.DV) * 128u;

    // The TMA warp decodes the CTA's first unit (blockIdx.x); later units come
    // from the call's unit counter.  Its lane 0 initialises the barriers,
    // publishes the unit and starts the copies the first S product needs (the
    // Q tile and K tile 0), so they are in flight while the other warps set up
    // the ones rows and TMEM.
    int4 mine = make_int4(0, 0, 0, 0);
    int split_first = 0, split_k = 1, units = 0;
    Unit w0;
    bool have0 = false;
    if (warp == WARP_TMA) {
        mine = find_item_load(p);
        const int4 hdr = *reinterpret_cast<const int4*>(p.ws);   // error, total_items, num_seqs, split_first
        split_k = p.ws->split_k;
        split_first = hdr.w;
        units = split_k > 1 ? split_first + (hdr.y - split_first) * split_k : hdr.y;
        have0 = int(blockIdx.x) < units && decode_unit(p, blockIdx.x, split_first, split_k, mine, w0);
        if (lane == 0) {
            mbar_init(BAR(B_QFULL), 1);
            for (int s = 0; s < NST; ++s) {
                mbar_init(BAR(B_KFULL + s), 1);
                mbar_init(BAR(B_VFULL + s), 1);
                mbar_init(BAR(B_KEMPTY + s), 1);
                mbar_init(BAR(B_VEMPTY + s), 1);
            }
            mbar_init(BAR(B_SFULL), 1);
            mbar_init(BAR(B_SFREE), 8);
            mbar_init(BAR(B_PFULL), 8);
            mbar_init(BAR(B_OFULL), 1);
            mbar_init(BAR(B_FINAL), 2);   // one commit per issuer
            mbar_init(BAR(B_QEMPTY), 1);
            mbar_init(BAR(B_OFREE), 8);
            for (int s = 0; s < 2; ++s) {
                mbar_init(BAR(B_IFULL + s), 1);
                mbar_init(BAR(B_IEMPTY + s), IEMPTY_COUNT);
            }
            *abort_flag = 0;
            fence_mbar_init();
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            volatile int* inf = INFO(0);
            inf[I_WORK] = have0 ? 1 : 0;
            if (have0) {
                inf[I_H] = w0.h;
                inf[I_Q0] = w0.q0;
                inf[I_SEGS] = w0.seg_s;
                inf[I_SEGE] = w0.seg_e;
                inf[I_KB0] = w0.kb0;
                inf[I_NKV] = w0.nkv;
                inf[I_SLOT] = w0.slot;
                inf[I_GRP] = w0.grp;
                inf[I_PARTS] = w0.parts;
            }
            mbar_arrive(BAR(B_IFULL + 0));
            // V^T copies start at token kb0 + j * BN, a multiple of 16: TMA needs
            // the innermost coordinate 16-byte aligned (checked in the checked build).
            if (have0 && VF_CHECKED_BUILD && (w0.kb0 & 15) != 0) {
                record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
                *abort_flag = 1;
            } else if (have0) {
                mbar_arrive_expect_tx(BAR(B_QFULL), QBYTES);
                tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, w0.h, w0.q0);
                mbar_arrive_expect_tx(BAR(B_KFULL + 0), KBYTES);
                tma_load_3d(sb + SM_K, &tmK, BAR(B_KFULL + 0), 0, w0.h, w0.kb0);
            }
        }
    }

    // Set-up sync on named barrier 1: the TMA warp only arrives (once the
    // barriers are initialised) and goes straight on with its copies; every
    // other warp also writes the ones rows and allocates TMEM, then waits.
    uint32_t tmem = 0;
    if (warp == WARP_TMA) {
        __syncwarp();
        __threadfence_block();
        named_bar_arrive<1, NUM_THREADS>();
    } else {
        // Rows DV..DV+15 of every V^T block hold E4M3 1.0 (0x38) for good:
        // the TMA boxes cover rows 0..DV-1 only.  (Uniform bytes: the swizzle
        // does not matter.)  The tensor core reads them through the async
        // proxy.
        const int t = threadIdx.x < 32 * WARP_TMA ? threadIdx.x : threadIdx.x - 32;
        for (int i = t; i < NST * 2 * 16 * 32; i += NUM_THREADS - 32) {
            const int blk = i / (16 * 32);
            const int wd = i - blk * (16 * 32);
            if (VF_IN(blk * VBLK + p.DV * 128 + 4 * wd, 4, NST * VBYTES, &p.ws->error))
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
        regs_decrease<REGS_PRODUCER_P>();
        if (warp == WARP_TMA) {
            // ------------------------------------------------ TMA producer
            // Units one after another: publish the unit in description slot
            // qi & 1 (once the unit two before has been used up), load its Q
            // once every S product of the previous unit is done, then its K/V
            // tiles through the ring; ring stage and phase count tiles across
            // units (g).  The whole warp decodes (one vote over the records);
            // lane 0 issues.
            int g = 0;            // K/V tiles whose copies were started
            int kq = 0;           // Q tiles started
            bool k_only = false;  // K of tile g started, its V not
            bool ok = !*abort_flag;
            Unit w = w0;
            bool have = have0;
            for (int qi = 0; ok && have; ++qi) {
                if (lane == 0) {
                    const int slot = qi & 1;
                    if (qi > 0) {
                        if (qi >= 2) ok = bwait(BAR(B_IEMPTY + slot), ((qi - 2) >> 1) & 1, abort_flag, err);
                        if (ok) {
                            volatile int* inf = INFO(slot);
                            inf[I_WORK] = 1;
                            inf[I_H] = w.h;
                            inf[I_Q0] = w.q0;
                            inf[I_SEGS] = w.seg_s;
                            inf[I_SEGE] = w.seg_e;
                            inf[I_KB0] = w.kb0;
                            inf[I_NKV] = w.nkv;
                            inf[I_SLOT] = w.slot;
                            inf[I_GRP] = w.grp;
                            inf[I_PARTS] = w.parts;
                            mbar_arrive(BAR(B_IFULL + slot));
                            if (VF_CHECKED_BUILD && (w.kb0 & 15) != 0) {
                                record_error(err, VITFP8_ERR_DEVICE_BOUNDS);
                                *abort_flag = 1;
                                ok = false;
                            } else if ((ok = bwait(BAR(B_QEMPTY), (qi - 1) & 1, abort_flag, err))) {
                                mbar_arrive_expect_tx(BAR(B_QFULL), QBYTES);
                                tma_load_3d(sb + SM_Q, &tmQ, BAR(B_QFULL), 0, w.h, w.q0);
                            }
                        }
                    }
                    if (ok) ++kq;
                    for (int j = 0; ok && j < w.nkv; ++j, ++g) {
                        const int s = g % NST;
                        const int key0 = w.kb0 + j * BN;
                        if (!(qi == 0 && j == 0)) {   // K tile 0 of the first unit went out at set-up
                            if (g >= NST && !(ok = bwait(BAR(B_KEMPTY + s), ((g / NST) - 1) & 1, abort_flag, err))) break;
                            mbar_arrive_expect_tx(BAR(B_KFULL + s), KBYTES);
                            tma_load_3d(sb + SM_K + s * KBYTES, &tmK, BAR(B_KFULL + s), 0, w.h, key0);
                        }
                        if (g >= NST && !(ok = bwait(BAR(B_VEMPTY + s), ((g / NST) - 1) & 1, abort_flag, err))) {
                            k_only = true;
                            break;
                        }
                        mbar_arrive_expect_tx(BAR(B_VFULL + s), vbytes);
                        tma_load_3d(sb + SM_V + s * VBYTES, &tmV, BAR(B_VFULL + s), key0, 0, w.h);
                        tma_load_3d(sb + SM_V + s * VBYTES + VBLK, &tmV, BAR(B_VFULL + s), key0 + HALF, 0, w.h);
                    }
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                // The next unit: every lane takes part in the record vote.
                int nu = 0;
                if (lane == 0) nu = int(gridDim.x) + atomicAdd(&p.ws->next_unit, 1);
                nu = __shfl_sync(0xFFFFFFFFu, nu, 0);
                have = nu < units && decode_unit(p, nu, split_first, split_k, mine, w);
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
                const uint32_t idS = make_idesc(0, BM, BN);      // 128 x 256 per S product
                // Descriptors are built once: within a 128-byte swizzled row a
                // 32-byte K step adds 2 to the encoded start address; a stage
                // adds its byte offset / 16.
                const uint64_t dQ = sw128_kmajor_desc(sb + SM_Q);
                const uint64_t dK0 = sw128_kmajor_desc(sb + SM_K);
                const uint32_t tS = tmem + TM_S;
                const int KS = p.KS;
                // Tile g (counted across units) uses ring stage s = g % NST in
                // phase kph = (g / NST) & 1; gpar = g & 1.
                int s = 0;
                uint32_t kph = 0, gpar = 0;
                bool first = true;
                bool ok = true;
                for (int qi = 0; ok; ++qi) {
                    const int slot = qi & 1;
                    if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                    if (!INFO(slot)[I_WORK]) break;
                    const int nkv = INFO(slot)[I_NKV];
                    if (!(ok = bwait(BAR(B_QFULL), qi & 1, abort_flag, err))) break;
                    for (int j = 0; j < nkv; ++j) {
                        // S(g) as soon as K_g is in and every softmax warp has read S(g-1).
                        if (!(ok = bwait(BAR(B_KFULL + s), kph, abort_flag, err))) break;
                        if (!first && !(ok = bwait(BAR(B_SFREE), gpar ^ 1u, abort_flag, err))) break;
                        tc_fence_after();
                        const uint64_t dk = dK0 + uint64_t(s * (KBYTES >> 4));
                        if (KS == 4) {
                            umma_f8_ss_k4(tS, dQ, dk, idS, 0u);
                        } else {
                            umma_f8(tS, dQ, dk, idS, 0u);
                            for (int kk = 1; kk < KS; ++kk)
                                umma_f8(tS, dQ + uint64_t(2 * kk), dk + uint64_t(2 * kk), idS, 1u);
                        }
                        tc_commit(BAR(B_SFULL));
                        tc_commit(BAR(B_KEMPTY + s));
                        first = false;
                        gpar ^= 1u;
                        if (++s == NST) {
                            s = 0;
                            kph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    tc_commit(BAR(B_QEMPTY));   // every S product of this unit read Q
                    mbar_arrive(BAR(B_IEMPTY + slot));
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
                const uint32_t tO = tmem + TM_O, tP = tmem + TM_P;
                int s = 0;
                uint32_t vph = 0, gpar = 0;   // as in the S issuer
                bool ok = true;
                for (int qi = 0; ok; ++qi) {
                    const int slot = qi & 1;
                    if (!(ok = bwait(BAR(B_IFULL + slot), (qi >> 1) & 1, abort_flag, err))) break;
                    if (!INFO(slot)[I_WORK]) break;
                    const int nkv = INFO(slot)[I_NKV];
                    for (int j = 0; j < nkv; ++j) {
                        // O += P(g) V_g: 256 keys in 8 steps of 32, keys 0..127 from
                        // V^T block 0 and P columns 0..31, keys 128..255 from block 1
                        // and P columns 32..63.  A unit's first product overwrites O,
                        // once the softmax has read the previous unit's O.
                        if (!(ok = bwait(BAR(B_VFULL + s), vph, abort_flag, err))) break;
                        if (!(ok = bwait(BAR(B_PFULL), gpar, abort_flag, err))) break;
                        if (j == 0 && qi > 0 && !(ok = bwait(BAR(B_OFREE), (qi - 1) & 1, abort_flag, err))) break;
                        tc_fence_after();
                        const uint64_t dv = dV0 + uint64_t(s * (VBYTES >> 4));
                        umma_f8_ts_k4(tO, tP, dv, idPV, j > 0 ? 1u : 0u);
                        umma_f8_ts_k4(tO, tP + 32u, dv + uint64_t(VBLK >> 4), idPV, 1u);
                        tc_commit(BAR(B_OFULL));
                        tc_commit(BAR(B_VEMPTY + s));
                        gpar ^= 1u;
                        if (++s == NST) {
                            s = 0;
                            vph ^= 1u;
                        }
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
        regs_increase<REGS_SOFTMAX_P>();
        const int half = lane >> 4;           // keys half*128 .. half*128+127 of each tile
        const int rbase = 32 * (warp & 3) + 16 * (warp >> 2);
        const int r = rbase + (lane & 15);    // row inside the query tile
        const uint32_t lane_off = uint32_t(rbase) << 16;
        const uint32_t tS = tmem + lane_off + TM_S;
        const uint32_t tO = tmem + lane_off + TM_O;
        const uint32_t tP = tmem + lane_off + TM_P;
        const float c = p.st->scale[0] * p.st->scale[1] * p.sm_scale * 1.4426950408889634f;
        const uint64_t c2 = f32x2_pack(c, c);
        const float scale_v = p.st->scale[2];
        const SoftmaxWarp sw{tS, tO, tP, sb + SM_BAR, c2, c, p.DV, abort_flag, err};
        int g = 0;
        bool ok = true;
        for (int qi = 0; ok; ++qi) {
            ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_IFULL + (qi & 1)), (qi >> 1) & 1, abort_flag, err));
            if (!ok) break;
            // The unit's description, broadcast from lane 0 so that the
            // compiler sees warp-uniform values (uniform datapath, fewer
            // registers in the tile loop).
            if (!__shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_WORK], 0)) break;
            const int seg_s = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_SEGS], 0);
            const int seg_e = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_SEGE], 0);
            const int kb0 = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_KB0], 0);
            const int nkv = __shfl_sync(0xFFFFFFFFu, INFO(qi & 1)[I_NKV], 0);
            float m_ref = 0.0f;
            for (int j = 0; j < nkv; ++j, ++g) {
                ok = softmax_tile(sw, kb0 + j * BN + half * HALF, seg_s, seg_e, j == 0, uint32_t(g) & 1u, m_ref);
                if (!ok) break;
            }
            if (ok) ok = __all_sync(0xFFFFFFFFu, bwait(BAR(B_OFULL), (g - 1) & 1, abort_flag, err));
            if (!ok) break;
            // ---- epilogue of the unit (its description is still in the slot)
            volatile int* inf = INFO(qi & 1);
            const int h = __shfl_sync(0xFFFFFFFFu, inf[I_H], 0);
            const int qrow = __shfl_sync(0xFFFFFFFFu, inf[I_Q0], 0) + r;   // packed token index of this row
            const bool row_valid = qrow < seg_e;
            const int parts = __shfl_sync(0xFFFFFFFFu, inf[I_PARTS], 0);
            tc_fence_after();
            if (parts == 1) {
                uint32_t lbits;   // both halves: a copy of l (column DV)
                uint32_t oa[32], ob[32], oc[16];
                tmem_ld_o80<OSPLIT>(tO, tO + uint32_t(p.DV), oa, ob, oc, lbits);
                // O is in registers: the next unit's first P.V may overwrite it.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_OFREE));
                const float oscale = scale_v / __uint_as_float(lbits);
                uint16_t* orow = p.out + (int64_t(qrow) * p.H + h) * p.D;
                const int cbase = half * OSPLIT;
                auto store8 = [&](int d0, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                  uint32_t a5, uint32_t a6, uint32_t a7) {
                    if (!row_valid || d0 + 8 > p.D) return;
                    if (!VF_IN((int64_t(qrow) * p.H + h) * p.D + d0, 8, p.out_elems, err)) return;
                    uint4 v;
                    v.x = cvt_bf16x2(__uint_as_float(a0) * oscale, __uint_as_float(a1) * oscale);
                    v.y = cvt_bf16x2(__uint_as_float(a2) * oscale, __uint_as_float(a3) * oscale);
                    v.z = cvt_bf16x2(__uint_as_float(a4) * oscale, __uint_as_float(a5) * oscale);
                    v.w = cvt_bf16x2(__uint_as_float(a6) * oscale, __uint_as_float(a7) * oscale);
                    *reinterpret_cast<uint4*>(orow + d0) = v;
                };
#pragma unroll
                for (int q = 0; q < 32; q += 8) {
                    store8(cbase + q, oa[q], oa[q + 1], oa[q + 2], oa[q + 3], oa[q + 4], oa[q + 5], oa[q + 6], oa[q + 7]);
                    store8(cbase + 32 + q, ob[q], ob[q + 1], ob[q + 2], ob[q + 3], ob[q + 4], ob[q + 5], ob[q + 6],
                           ob[q + 7]);
                }
                store8(cbase + 64, oc[0], oc[1], oc[2], oc[3], oc[4], oc[5], oc[6], oc[7]);
                store8(cbase + 72, oc[8], oc[9], oc[10], oc[11], oc[12], oc[13], oc[14], oc[15]);
            } else {
                SplitOut so;
                so.part = p.split_part;
                so.cnt = p.split_cnt;
                so.out = p.out + (int64_t(qrow) * p.H + h) * p.D;
                so.err = err;
                so.out_off = (int64_t(qrow) * p.H + h) * p.D;
                so.out_elems = p.out_elems;
                so.D = p.D;
                so.DV = p.DV;
                split_part_epilogue(so, tO, row_valid, half, m_ref, scale_v, inf[I_SLOT], inf[I_GRP], parts, true,
                                    abort_flag, smem + SM_LAST, BAR(B_OFREE));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_IEMPTY + (qi & 1)));
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

// Work list: one record per segment, segments sorted longest first (when
// there are at most 2048; in cu_seqlens order otherwise), items per segment =
// ceil(L / rows_per_item) * H, each record's first_item the items of all
// records before it (a block-wide scan, 1024 records per step).
//
// Key-range split (split_bn > 0): N items on nsm SMs leave r = N mod nsm items
// for a last wave that would hold the GPU for a whole item while most SMs
// idle.  When r <= nsm / 2, each of those r items is cut into k = nsm / r
// parts (at most kSplitMaxK, at most kSplitMaxParts CTAs, and no more parts
// than the item has key tiles of split_bn keys), one CTA per part.
__global__ void attn_plan_kernel(const int32_t* __restrict__ cu, int nseq, int T, int H,
                                 int rows_per_item, int nsm, int split_bn, WsHeader* ws,
                                 SegRec* rec, int32_t* split_cnt) {
    __shared__ int bad;
    __shared__ int warp_sum[32];
    __shared__ int carry;
    if (threadIdx.x == 0) {
        ws->error = 0;
        bad = (cu[0] != 0 || cu[nseq] != T) ? 1 : 0;
        carry = 0;
    }
    if (split_cnt != nullptr)
        for (int i = threadIdx.x; i < kSplitMaxParts; i += blockDim.x) split_cnt[i] = 0;
    __syncthreads();
    for (int b = threadIdx.x; b < nseq; b += blockDim.x)
        if (cu[b + 1] < cu[b]) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) {
            ws->total_items = 0;
            ws->num_seqs = nseq;
            ws->split_first = 0;
            ws->split_k = 1;
            ws->next_unit = 0;
            record_error(&ws->error, VITFP8_ERR_BAD_SEQLENS);
        }
        return;
    }
    for (int b = threadIdx.x; b < nseq; b += blockDim.x) {
        const int Lb = cu[b + 1] - cu[b];
        int rank = b;
        if (nseq <= 2048) {
            rank = 0;
            for (int b2 = 0; b2 < nseq; ++b2) {
                const int L2 = cu[b2 + 1] - cu[b2];
                rank += (L2 > Lb) || (L2 == Lb && b2 < b);
            }
        }
        if (VF_IN(rank, 1, nseq, &ws->error))
            *reinterpret_cast<int4*>(rec + rank) =
                make_int4(0, cu[b], cu[b + 1], (Lb + rows_per_item - 1) / rows_per_item);
    }
    __syncthreads();
    // first_item: exclusive scan of nq * H over the records, 1024 at a time.
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int base = 0; base < nseq; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = i < nseq ? rec[i].nq * H : 0;
        int x = v;   // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < nw) warp_sum[lane] = w;   // inclusive prefix of warp totals
        }
        __syncthreads();
        const int before = carry + (wid > 0 ? warp_sum[wid - 1] : 0) + x - v;
        if (i < nseq) rec[i].first_item = before;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) carry = before + v;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int N = carry;
        int sfirst = N, sk = 1;
        const int r = nsm > 0 ? N % nsm : 0;
        if (split_bn > 0 && split_cnt != nullptr && r > 0 && 2 * r <= nsm) {
            int k = min(min(nsm / r, kSplitMaxK), kSplitMaxParts / r);
            // Every part needs a key tile of its own: the segments of items N-r..N-1.
            for (int b = nseq - 1; b >= 0; --b) {
                if (!VF_IN(b, 1, nseq, &ws->error)) break;
                const SegRec R = rec[b];
                if (R.nq == 0) continue;
                if (R.first_item + R.nq * H <= N - r) break;
                k = min(k, (R.seg_e - (R.seg_s & ~15) + split_bn - 1) / split_bn);
            }
            if (k >= 2) {
                sfirst = N - r;
                sk = k;
            }
        }
        ws->total_items = N;
        ws->num_seqs = nseq;
        ws->split_first = sfirst;
        ws->split_k = sk;
        ws->next_unit = 0;
    }
}

// ---------------------------------------------------------------- host side

namespace {
using EncodeFn = decltype(&cuTensorMapEncodeTiled);

// cuTensorMapEncodeTiled from the driver, looked up once per process (the
// function-local static is initialised once, thread-safely); null if the
// driver does not provide it.
EncodeFn get_encode_fn() {
    static const EncodeFn fn = []() -> EncodeFn {
        cudaDriverEntryPointQueryResult q;
        void* ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeFn>(ptr);
        return nullptr;
    }();
    return fn;
}

bool make_map_3d_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {stride1, stride2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The kernels' dynamic shared memory (above the 48 KB default) is opted into
// once per device: the attribute belongs to the current device.
PerDeviceOnce g_smem_attr;
}  // namespace

cudaError_t launch_attn_plan(const int32_t* cu, int nseq, int T, int H, int rows_per_item,
                             int nsm, int split_bn, void* ws, cudaStream_t s) {
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    int32_t* cnt = split_bn > 0 ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) +
                                                             ws_split_cnt_offset(nseq))
                                : nullptr;
    attn_plan_kernel<<<1, 1024, 0, s>>>(cu, nseq, T, H, rows_per_item, nsm, split_bn, hdr,
                                        reinterpret_cast<SegRec*>(hdr + 1), cnt);
    return cudaGetLastError();
}

vitfp8_status launch_attn_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                              const vitfp8_scale_state* st, const int32_t* cu, int nseq, int max_seqlen,
                              int T, int H, int D, int Dp, int64_t Tv, float sm_scale, uint16_t* out,
                              void* ws, int kernel, cudaStream_t s) {
    using namespace fa;
    if (kernel < kAttnAuto || kernel > kAttnTwoTilePersistent) return VITFP8_ERR_INVALID_ARG;
    const int DV = (D + 15) & ~15;
    int dev = -1, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return VITFP8_ERR_CUDA;
    if (kernel == kAttnAuto) kernel = attn_fp8_kernel_for(nseq, max_seqlen, T, H, nsm);
    // Q boxes of 128 rows and V^T boxes of 128 keys for every kernel; K boxes
    // of one key tile (256 keys, 128 for the two-tile kernel).
    CUtensorMap mq, mk, mv;
    if (!make_map_3d_u8(&mq, q8, uint64_t(Dp), uint64_t(H), uint64_t(T), uint64_t(Dp),
                        uint64_t(H) * Dp, 128, 1, BM) ||
        !make_map_3d_u8(&mk, k8, uint64_t(Dp), uint64_t(H), uint64_t(T), uint64_t(Dp),
                        uint64_t(H) * Dp, 128, 1, kernel >= kAttnTwoTile ? 128u : uint32_t(BN)) ||
        !make_map_3d_u8(&mv, v8t, uint64_t(Tv), uint64_t(Dp), uint64_t(H), uint64_t(Tv),
                        uint64_t(Tv) * Dp, HALF, uint32_t(DV), 1))
        return VITFP8_ERR_CUDA;

    if (!g_smem_attr.run(dev, [] {
            return cudaFuncSetAttribute(attn_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        SMEM_BYTES) == cudaSuccess &&
                   cudaFuncSetAttribute(attn_fp8_persistent_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) == cudaSuccess;
        }))
        return VITFP8_ERR_CUDA;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    AttnParams prm;
    prm.cu = cu;
    prm.rec = reinterpret_cast<const SegRec*>(hdr + 1);
    prm.ws = hdr;
    prm.st = st;
    prm.out = out;
    prm.split_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ws_split_cnt_offset(nseq));
    prm.split_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + ws_split_part_offset(nseq));
    prm.nseq = nseq;
    prm.T = T;
    prm.H = H;
    prm.D = D;
    prm.Dp = Dp;
    prm.DV = DV;
    prm.KS = (D + 31) / 32;
    prm.sm_scale = sm_scale;
    prm.out_elems = int64_t(T) * H * D;
    if (kernel >= kAttnTwoTile)
        return launch_attn_fp8_2tile(mq, mk, mv, prm, nsm, kernel == kAttnTwoTilePersistent, s);

    if (launch_attn_plan(cu, nseq, T, H, ROWS_PER_ITEM, nsm, BN, ws, s) != cudaSuccess)
        return VITFP8_ERR_CUDA;
    // Units (work items, or parts of split items) are at most
    // (T / 128 + nseq) * H + kSplitMaxParts; CTAs without a unit return at once.
    const long long max_units = (long long)((T + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM + nseq) * H + kSplitMaxParts;
    if (max_units > 0x7FFFFFFFLL) return VITFP8_ERR_UNSUPPORTED;
    if (kernel == kAttnPersistent) {
        // One CTA per SM walking the units, so a unit's set-up and first loads
        // overlap the previous unit's last tiles (worth it for short segments).
        const unsigned grid = unsigned(max_units < nsm ? max_units : nsm);
        attn_fp8_persistent_kernel<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    } else {
        attn_fp8_kernel<<<unsigned(max_units), NUM_THREADS, SMEM_BYTES, s>>>(mq, mk, mv, prm);
    }
    return cudaGetLastError() == cudaSuccess ? VITFP8_OK : VITFP8_ERR_CUDA;
}

}  // namespace vitfp8
