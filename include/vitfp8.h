/*
 * vitfp8 -- FP8 ViT-encoder attention for one GB300 (sm_103a).  C ABI.
 *
 * The hot path of one ViT-encoder attention layer, as the pages describe it
 * ("FP8 ViT Encoder Attention", vLLM docs; "FP8 vision encoder attention",
 * Sonar):
 *
 *   1. per-tensor amax of Q, K and V kept in a 16-entry circular history
 *      (dynamic scaling) -- or static per-layer scales from a scale file;
 *   2. on-the-fly FP8 (E4M3) quantization of Q, K and V fused with
 *      un-padding into a packed variable-length layout;
 *   3. non-causal variable-length attention over packed multi-image batches
 *      delimited by cu_seqlens, with FP8 QK^T and FP8 P.V on tensor cores and
 *      a bf16 output.
 *
 * Conventions for every entry point below:
 *
 *   - Pointers named d_* and all tensor pointers are DEVICE pointers; h_* are
 *     HOST pointers.  The caller allocates and frees every buffer (sources,
 *     codes, outputs, state, workspace).  The library never allocates or
 *     frees memory on these calls.  Its only process-wide state is set-up
 *     that belongs to a device and is done once per device, under a lock, on
 *     the first call that needs it: the attention kernels' opt-in to more
 *     than 48 KB of shared memory, the driver's tensor-map encoder (looked
 *     up once per process), and the device address of the scratch array of
 *     vitfp8_attn_varlen_noalloc.  Every entry point may be called from
 *     several host threads at once and for several devices in one process;
 *     calls on one stream run in order, calls on different streams that
 *     share a buffer must be ordered by the caller.
 *   - All work is enqueued asynchronously on `stream`; nothing synchronises
 *     with the host except vitfp8_get_device_error /
 *     vitfp8_get_workspace_error, which synchronise `stream`.
 *   - Argument errors are detected on the host and returned before any launch
 *     (VITFP8_ERR_INVALID_ARG / VITFP8_ERR_UNSUPPORTED).  A failed launch
 *     returns VITFP8_ERR_CUDA.  Errors found on the device (malformed
 *     cu_seqlens, a bounded wait that timed out) are recorded in a device
 *     error word and read back with the two *_get_*_error calls.
 *   - Nothing aborts, traps or throws across this boundary.
 *   - bf16 tensors are passed as vitfp8_bf16 (the raw 16-bit pattern).
 *   - Tensors must be 16-byte aligned; sizes and strides are in ELEMENTS.
 */
#ifndef VITFP8_H
#define VITFP8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t vitfp8_bf16; /* bfloat16 bit pattern */

typedef enum vitfp8_status {
    VITFP8_OK = 0,
    VITFP8_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad size or stride */
    VITFP8_ERR_UNSUPPORTED = 2,    /* valid request outside what the kernels cover (e.g. D > 128) */
    VITFP8_ERR_CUDA = 3,           /* a CUDA runtime / driver call failed */
    VITFP8_ERR_DEVICE_TIMEOUT = 4, /* device: a bounded wait expired; the kernel returned early */
    VITFP8_ERR_DEVICE_BOUNDS = 5,  /* device (checked build): an index fell outside its buffer and was skipped */
    VITFP8_ERR_BAD_SEQLENS = 6,    /* device: cu_seqlens not 0 = c0 <= c1 <= ... <= c_B = T */
    VITFP8_ERR_WORKSPACE = 7       /* workspace missing or smaller than vitfp8_attn_workspace_size */
} vitfp8_status;

#define VITFP8_RING 16          /* amax history length ("16-entry circular buffer") */
#define VITFP8_E4M3_MAX 448.0f  /* largest finite E4M3 value */
#define VITFP8_MAX_HEAD_DIM 128 /* largest head dim the attention kernels take */

/*
 * One layer's FP8 scale state, DEVICE-resident, one per attention layer.
 *
 * Source: "FP8 ViT Encoder Attention", Usage -- a 16-entry circular buffer of
 * observed Q/K/V amax values drives per-forward scale updates; Calibrate-Once
 * and Scale File Format -- static per-layer q/k/v values.
 *
 * Index t in the [3] arrays is 0 = q, 1 = k, 2 = v.  A "scale value" A is an
 * amax-like magnitude: dequantisation factor scale = A/448, quantisation
 * multiplier inv_scale = 448/A (each one IEEE float32 division).  If A == 0
 * both are 1.  The fields amax_bits and blocks_done are reduction scratch
 * owned by vitfp8_amax_update; they are zero between calls.
 */
typedef struct vitfp8_scale_state {
    float    hist[3][VITFP8_RING]; /* amax ring per tensor; empty slots hold 0 */
    int32_t  pos;                  /* slot the next forward writes */
    int32_t  count;                /* filled slots, <= 16 */
    int32_t  mode;                 /* 0 dynamic, 1 static, 2 dynamic with delayed scaling */
    int32_t  dev_error;            /* first device-detected vitfp8_status, 0 if none */
    float    amax_ref[3];          /* A_t: ring maximum (dynamic) or the static value */
    float    scale[3];             /* A_t / 448 */
    float    inv_scale[3];         /* 448 / A_t */
    float    amax_cur[3];          /* amax of the latest dynamic forward */
    uint32_t amax_bits[3];         /* scratch: running max of |x| as bf16 magnitude bits */
    uint32_t blocks_done;          /* scratch: finished blocks of the current amax launch */
} vitfp8_scale_state;

/*
 * Where the valid bf16 source rows of Q, K or V live ("un-padding").
 *
 * padded = 1: a padded batch -- segment b's token i sits at row b*s_max + i;
 *             rows i >= L_b are padding and are never read.
 * padded = 0: packed rows -- segment b's token i sits at row cu_seqlens[b]+i.
 * Element (row, h, d) is at row*token_stride + h*head_stride + d (elements);
 * d is contiguous.  token_stride and head_stride must be multiples of 8 so
 * that every 8-element vector is 16-byte aligned (e.g. a view into a fused
 * [T, 3, H, D] QKV buffer has token_stride 3*H*D).
 */
typedef struct vitfp8_src_layout {
    int32_t padded;
    int32_t reserved;
    int64_t s_max;
    int64_t token_stride;
    int64_t head_stride;
} vitfp8_src_layout;

/* Human-readable name of a status code (static string, never NULL). */
const char* vitfp8_status_string(vitfp8_status s);

/* Library ABI version (major*100 + minor). */
int32_t vitfp8_version(void);

/*
 * Reset a state to dynamic mode with an empty ring (all slots 0, pos 0,
 * count 0, scale = inv_scale = 1, dev_error 0, scratch 0).
 * d_state: device pointer to one vitfp8_scale_state (4-byte aligned).
 */
vitfp8_status vitfp8_scale_state_init(vitfp8_scale_state* d_state, cudaStream_t stream);

/*
 * Switch a state to static mode with the scale-file values q, k, v
 * ("FP8 ViT Encoder Attention", Scale File Format: e.g. 224, 198, 210).
 * Each value must be finite and > 0 (else VITFP8_ERR_INVALID_ARG, nothing
 * launched).  Sets amax_ref = value, scale = value/448, inv_scale = 448/value.
 */
vitfp8_status vitfp8_set_static_scales(vitfp8_scale_state* d_state, float q, float k, float v,
                                       cudaStream_t stream);

/*
 * Order of the ring update in dynamic mode.  delayed = 0 (the default after
 * init; mode 0): push the forward's amax, then take the scale from the ring
 * including it, so the forward never saturates.  delayed != 0 (mode 2,
 * delayed scaling): take the scale from the ring the earlier forwards left,
 * then push -- the forward is quantized with its predecessors' history (the
 * first forward with scale 1) and may saturate at +-448.  The pages describe
 * the 16-entry ring ("FP8 ViT Encoder Attention", Usage) but not this order.
 * A static state is left unchanged.  The ring contents are the same in both
 * orders; only amax_ref / scale / inv_scale lag by one forward.
 */
vitfp8_status vitfp8_set_ring_order(vitfp8_scale_state* d_state, int32_t delayed,
                                    cudaStream_t stream);

/*
 * Dynamic scaling, one forward ("FP8 ViT Encoder Attention", Usage; Sonar,
 * Enable FP8 attention): amax of q, k and v over the valid tokens (all heads,
 * d < D), pushed into the 16-entry ring (push-then-scale), then
 * amax_ref = max(ring), scale and inv_scale recomputed (in mode 2 the
 * scale is taken before the push; see vitfp8_set_ring_order).  One launch covers
 * all three tensors; the last block to finish updates the ring.
 * In static mode the launch returns without touching the state (a no-op).
 *
 * q, k, v:        bf16 sources, layout given by *h_layout (host pointer).
 * d_cu_seqlens:   int32[num_seqs + 1] on the device, 0 = c0 <= ... <= c_B = total_tokens.
 * total_tokens:   T = c_B (host copy); T == 0 or num_seqs == 0 is a no-op.
 * H, D:           heads and head dim; D % 8 == 0, 8 <= D <= 256.
 * Amax follows fmax semantics: NaN ignored, +inf propagates.
 * Concurrent calls on the same state race (the scratch fields are shared).
 */
vitfp8_status vitfp8_amax_update(vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                 const vitfp8_bf16* k, const vitfp8_bf16* v,
                                 const vitfp8_src_layout* h_layout, const int32_t* d_cu_seqlens,
                                 int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t D,
                                 cudaStream_t stream);

/*
 * Data-parallel dynamic scaling, step 1 of 3.  The amax of the pages is one
 * value per tensor over the whole batch ("FP8 ViT Encoder Attention", Usage);
 * when the batch's segments are spread over several GPUs, each rank computes
 * the amax of its own tokens here, the ranks combine the four floats with an
 * all-reduce(MAX) (step 2, the caller's collective), and every rank pushes
 * the result with vitfp8_ring_push (step 3), so all rings stay identical to
 * the single-GPU ring of the whole batch.  On one GPU,
 * vitfp8_amax_local + vitfp8_ring_push == vitfp8_amax_update.
 *
 * Arguments as for vitfp8_amax_update, plus
 *   d_vals: device float[4] (4-byte aligned), written on the stream with
 *           (amax_q, amax_k, amax_v, 1) -- or (0, 0, 0, 0) when this rank has
 *           no tokens (T == 0 or num_seqs == 0) or the state is static.
 * The ring, pos, count and the scales are not changed; amax_cur gets the local amax.
 */
vitfp8_status vitfp8_amax_local(vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                const vitfp8_bf16* k, const vitfp8_bf16* v,
                                const vitfp8_src_layout* h_layout, const int32_t* d_cu_seqlens,
                                int32_t num_seqs, int32_t total_tokens, int32_t H, int32_t D,
                                float* d_vals, cudaStream_t stream);

/*
 * Data-parallel dynamic scaling, step 3 of 3: push (d_vals[0..2]) into the
 * ring and recompute amax_ref, scale and inv_scale exactly as
 * vitfp8_amax_update does -- if d_vals[3] > 0 (some rank had tokens).
 * No-op in static mode.  d_vals: device float[4], e.g. after all-reduce(MAX).
 */
vitfp8_status vitfp8_ring_push(vitfp8_scale_state* d_state, const float* d_vals,
                               cudaStream_t stream);

/*
 * Quantize + un-pad q, k and v in ONE launch ("FP8 ViT Encoder Attention",
 * intro and note: Q/K/V quantized on the fly before the attention call,
 * "quantization kernel launches + un-padding").
 *
 * code = E4M3(float32(x) * inv_scale[t]), round to nearest even, saturating
 * to +-448, NaN -> NaN code; entries d in [D, D_pad) are written as 0x00.
 *
 * Outputs (device, caller-allocated):
 *   q8, k8: uint8 [T][H][D_pad]   packed token order (row t*H + h).
 *   v8t:    uint8 [H][D_pad][Tv]  V transposed per head, tokens contiguous,
 *           Tv = vitfp8_vt_stride(T); tokens in [T, Tv) are written as 0x00.
 * D_pad: multiple of 16, D <= D_pad <= 256.
 */
vitfp8_status vitfp8_quantize_unpad(const vitfp8_scale_state* d_state, const vitfp8_bf16* q,
                                    const vitfp8_bf16* k, const vitfp8_bf16* v,
                                    const vitfp8_src_layout* h_layout,
                                    const int32_t* d_cu_seqlens, int32_t num_seqs,
                                    int32_t total_tokens, int32_t H, int32_t D, int32_t D_pad,
                                    uint8_t* q8, uint8_t* k8, uint8_t* v8t, cudaStream_t stream);

/* Token stride Tv of the transposed V code buffer: T rounded up to 16. */
int64_t vitfp8_vt_stride(int32_t total_tokens);

/* Bytes of device workspace vitfp8_attn_varlen(_bf16) needs for num_seqs segments. */
size_t vitfp8_attn_workspace_size(int32_t num_seqs);

/*
 * FP8 variable-length non-causal attention ("FP8 ViT Encoder Attention",
 * intro, Performance; Sonar, Requirements: packed variable-length batches,
 * per-tensor FP8).
 *
 * For each segment b (tokens c_b .. c_{b+1}-1), head h and query i of b:
 *   s_ij = (q8_i . k8_j) * scale_q * scale_k * sm_scale   over keys j in b only,
 *   softmax in fp32 (online), P requantized to E4M3 (relative to a
 *   power-of-two reference) for an FP8 P.V tensor-core product,
 *   o_i = (sum_j P_ij v8_j) * scale_v / sum_j p_ij, rounded to bf16.
 * No query attends across a cu_seqlens boundary.
 *
 * q8, k8:  uint8 [T][H][D_pad] E4M3 codes; v8t: uint8 [H][D_pad][Tv] (as
 *          written by vitfp8_quantize_unpad).
 * d_state: scales read on the device (scale[0..2]).
 * max_seqlen: host upper bound of the segment lengths (>= every L_b).
 * D: 8..128, D % 8 == 0; D_pad % 16 == 0, D <= D_pad <= 128.
 * sm_scale: softmax scale, normally 1/sqrt(D); finite and > 0.
 * out: bf16 [T][H][D].
 * d_workspace: >= vitfp8_attn_workspace_size(num_seqs) bytes (about 14 MB),
 *          16-byte aligned; holds the (longest-first) work list, an error
 *          word and the partial results of a key-range split.  Calls sharing
 *          one workspace must be stream-ordered.
 *
 * Scheduling (vitfp8_attn_kernel_for picks one of four kernels; all compute
 * the attention above):
 *  - VITFP8_ATTN_UNIT: one CTA per 128-query tile of a (segment, head).  When
 *    the tiles leave a last wave that fills at most half the GPU, the key range
 *    of each of those tiles is split over up to 4 units, and the unit that
 *    finishes last combines the parts by exact powers of two (same numerics up
 *    to the fp32 summation order).
 *  - VITFP8_ATTN_PERSISTENT: the same units run by one CTA per SM (for short
 *    segments); the same bits as VITFP8_ATTN_UNIT.
 *  - VITFP8_ATTN_TWO_TILE: one CTA per 256-query unit (two 128-row tiles
 *    sharing each key tile), for long segments whose units fill the GPU's
 *    waves well.  Its reference moves at 128-key boundaries, so about 1 % of
 *    the outputs can differ from the other kernels' in the last bf16 bit.
 *  - VITFP8_ATTN_TWO_TILE_PERSISTENT: the same units run by one CTA per SM
 *    (for segments of up to 6144 tokens); the same bits as
 *    VITFP8_ATTN_TWO_TILE.
 * The result is deterministic for a given input, max_seqlen and GPU.
 */
vitfp8_status vitfp8_attn_varlen(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                                 const vitfp8_scale_state* d_state, const int32_t* d_cu_seqlens,
                                 int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                 int32_t H, int32_t D, int32_t D_pad, float sm_scale,
                                 vitfp8_bf16* out, void* d_workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* FP8 attention kernels (vitfp8_attn_varlen_kernel's `kernel`). */
#define VITFP8_ATTN_AUTO 0       /* vitfp8_attn_kernel_for decides */
#define VITFP8_ATTN_UNIT 1       /* one CTA per 128-query work item */
#define VITFP8_ATTN_PERSISTENT 2 /* one CTA per SM walking the work items */
#define VITFP8_ATTN_TWO_TILE 3   /* one CTA per 256-query unit */
#define VITFP8_ATTN_TWO_TILE_PERSISTENT 4 /* the 256-query units run by one CTA per SM */

/*
 * vitfp8_attn_varlen with the kernel named by `kernel` (one of the
 * VITFP8_ATTN_* values; VITFP8_ATTN_AUTO is vitfp8_attn_varlen itself).
 * Every kernel takes every valid input; the choice only changes speed and,
 * for VITFP8_ATTN_TWO_TILE, the last bit of some outputs.  Errors as for
 * vitfp8_attn_varlen, plus VITFP8_ERR_INVALID_ARG for an unknown kernel.
 */
vitfp8_status vitfp8_attn_varlen_kernel(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                                        const vitfp8_scale_state* d_state, const int32_t* d_cu_seqlens,
                                        int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                        int32_t H, int32_t D, int32_t D_pad, float sm_scale,
                                        vitfp8_bf16* out, void* d_workspace, size_t workspace_bytes,
                                        int32_t kernel, cudaStream_t stream);

/*
 * The kernel vitfp8_attn_varlen runs for these sizes on a GPU with num_sms
 * SMs (host only, no device call).  With w = H (T + 128 num_seqs) / 256 /
 * num_sms, the estimated waves of 256-query units:
 *  - a two-tile kernel when w >= 2 and either max_seqlen < 2048 or
 *    ceil(w) / w <= 1.12 (the last wave nearly full): the persistent one
 *    (VITFP8_ATTN_TWO_TILE_PERSISTENT) when max_seqlen <= 6144, else
 *    VITFP8_ATTN_TWO_TILE;
 *  - else VITFP8_ATTN_PERSISTENT when max_seqlen <= 6144 and the 128-query
 *    items, (ceil(T / 128) + num_seqs) H, are more than num_sms;
 *  - else VITFP8_ATTN_UNIT (also for non-positive sizes).
 */
int32_t vitfp8_attn_kernel_for(int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens, int32_t H,
                               int32_t num_sms);

/*
 * BF16 variable-length non-causal attention, the comparison path of
 * "FP8 ViT Encoder Attention", Performance (the BF16 column of the kernel
 * and encoder tables): the same segment-masked attention as
 * vitfp8_attn_varlen, computed from the bf16 inputs directly, with no scales
 * and no quantization step.
 *
 * For each segment b, head h and query i of b:
 *   s_ij = (q_i . k_j) * sm_scale over keys j in b only (BF16 x BF16 -> fp32
 *   on the tensor cores), online softmax in fp32, P rounded to bf16 for the
 *   P.V product, o_i = (sum_j P_ij v_j) / sum_j P_ij (fp32 sum of the
 *   rounded weights, as in vitfp8_attn_varlen), rounded to bf16.
 *
 * q, k, v: bf16 [T][H][D], packed token order, rows contiguous (device).
 * D: 8..128, D % 8 == 0.  max_seqlen, sm_scale, out and d_workspace as for
 * vitfp8_attn_varlen (the same workspace size).  Scheduling as there, without
 * the key-range split: a persistent kernel for max_seqlen <= 6144 and more
 * than one wave of work items, one CTA per work item otherwise (same bits).
 * Errors: VITFP8_ERR_INVALID_ARG for bad sizes, null or misaligned (16-byte)
 * pointers; VITFP8_ERR_UNSUPPORTED for D > 128; VITFP8_ERR_WORKSPACE for a
 * missing or short workspace; malformed cu_seqlens and timed-out waits are
 * recorded in the workspace error word (vitfp8_get_workspace_error).
 */
vitfp8_status vitfp8_attn_varlen_bf16(const vitfp8_bf16* q, const vitfp8_bf16* k,
                                      const vitfp8_bf16* v, const int32_t* d_cu_seqlens,
                                      int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
                                      int32_t H, int32_t D, float sm_scale, vitfp8_bf16* out,
                                      void* d_workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/* Largest num_seqs vitfp8_attn_varlen_noalloc accepts. */
#define VITFP8_NOALLOC_MAX_SEQS 4096

/*
 * vitfp8_attn_varlen without a workspace argument: it allocates nothing and
 * needs nothing allocated by the caller beyond the inputs and the output.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot allocate device memory -- e.g. a plugin handed only raw input/output
 * pointers and no allocator, a serving host whose device memory pool is fixed
 * at start-up, or a latency-critical loop that cannot afford the device
 * synchronisation that cudaMalloc may cause.
 *
 * Arguments, layouts and the computation are exactly those of
 * vitfp8_attn_varlen.  The workspace (work list, error word and the partial
 * results of a key-range split) lives instead in a fixed device array inside
 * the library (about 14 MB; every GPU that loads the library keeps it until
 * the process exits), sized for at most VITFP8_NOALLOC_MAX_SEQS
 * segments: num_seqs above that returns VITFP8_ERR_UNSUPPORTED without
 * launching.  The first call on each device looks up that array's device
 * address (cudaGetSymbolAddress) with the device current; make that first
 * call before any stream capture.  The address is kept for the rest of the
 * process: after a cudaDeviceReset (or anything else that destroys the
 * device's primary context) the library's device code is loaded anew and the
 * kept address is stale, so do not call this entry point on that device
 * again in the same process.  Every call on a device shares the one
 * array and rewrites all of it that it reads, so nothing carries over between
 * calls; calls that overlap on the GPU (different streams, or different
 * host threads, without ordering) race on it.  Device-detected errors
 * (malformed cu_seqlens, a timed-out wait) leave the output unwritten and are
 * not reported by this entry point; use vitfp8_attn_varlen with a workspace
 * to read them.
 */
vitfp8_status vitfp8_attn_varlen_noalloc(const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t,
                                         const vitfp8_scale_state* d_state,
                                         const int32_t* d_cu_seqlens, int32_t num_seqs,
                                         int32_t max_seqlen, int32_t total_tokens, int32_t H,
                                         int32_t D, int32_t D_pad, float sm_scale, vitfp8_bf16* out,
                                         cudaStream_t stream);

/*
 * Device error word of a state: *h_out = first vitfp8_status recorded by a
 * kernel that used d_state (0 if none).  Synchronises `stream`.  h_out: host.
 */
vitfp8_status vitfp8_get_device_error(const vitfp8_scale_state* d_state, int32_t* h_out,
                                      cudaStream_t stream);

/* Same for an attention workspace.  Synchronises `stream`. */
vitfp8_status vitfp8_get_workspace_error(const void* d_workspace, int32_t* h_out,
                                         cudaStream_t stream);

/*
 * Failure-detection self-test: one warp runs the bounded mbarrier wait that
 * every role of the attention kernels uses, on a barrier nothing arrives on.
 * After the wait's limit (about 0.5 s) the kernel records
 * VITFP8_ERR_DEVICE_TIMEOUT in the workspace error word (cleared at launch)
 * and returns; read it with vitfp8_get_workspace_error.  Nothing traps,
 * faults or hangs, and the context stays usable.
 * d_workspace: at least vitfp8_attn_workspace_size(0) bytes, 4-byte aligned.
 */
vitfp8_status vitfp8_selftest_bounded_wait(void* d_workspace, size_t workspace_bytes,
                                          cudaStream_t stream);

/*
 * Calibrate once, on the device ("FP8 ViT Encoder Attention", Calibrate-Once,
 * Reuse Workflow; Scale File Format; "FP8 vision encoder attention" (Sonar),
 * Create static scales): after the calibration forwards (16 on the pages) of
 * a layer in dynamic mode, take each tensor's learned scale -- its ring
 * maximum A, whatever the ring order -- and the value the scale file saves,
 * float32(A) * float32(margin) (one float32 multiply; the pages' default
 * margin is 1.5).
 *
 * d_dynamic: the calibrated state (device, read only except its error word).
 * margin: finite, > 0 (else VITFP8_ERR_INVALID_ARG before any launch).
 * d_saved: optional device float[3], receives the saved values (q, k, v),
 *   which a caller copies back to write the scale file.
 * d_static: optional device state, set to static mode with the saved values
 *   exactly as vitfp8_set_static_scales would; must not be d_dynamic.
 * A tensor whose ring holds no amax (A == 0) has no valid static scale: the
 * dynamic state's error word records VITFP8_ERR_INVALID_ARG (read it with
 * vitfp8_get_device_error) and d_static is left unchanged.  Stream-ordered,
 * one launch, no host synchronisation.
 */
vitfp8_status vitfp8_calibrated_scales(const vitfp8_scale_state* d_dynamic, float margin,
                                       float* d_saved, vitfp8_scale_state* d_static,
                                       cudaStream_t stream);

/*
 * 1 if this library was compiled as the checked build (-DVITFP8_CHECKED),
 * else 0.  In the checked build every global- and shared-memory index the
 * kernels compute is compared with the extent its arguments imply (sources
 * by their layout, codes [T, H, D_pad] and [H, D_pad, Tv], output [T, H, D],
 * cu_seqlens and the work list by num_seqs); an index outside records
 * VITFP8_ERR_DEVICE_BOUNDS in the call's device error word (the scale
 * state's for amax and quantization, the workspace's for attention) and the
 * access is skipped.  Nothing traps.  The normal build has no checks.
 */
int32_t vitfp8_checked_build(void);

/*
 * Self-test of that bounds check: one thread asks the check whether element
 * 16 of a 16-element buffer may be accessed (the buffer is never touched).
 * The checked build records VITFP8_ERR_DEVICE_BOUNDS in the workspace error
 * word (cleared at launch); the normal build records nothing.  Read it with
 * vitfp8_get_workspace_error.  d_workspace: at least
 * vitfp8_attn_workspace_size(0) bytes, 4-byte aligned.
 */
vitfp8_status vitfp8_selftest_bounds_check(void* d_workspace, size_t workspace_bytes,
                                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VITFP8_H */
