// vitfp8_attn_varlen_noalloc: the FP8 varlen attention entry point for callers
// that cannot allocate device memory.
//
// vitfp8_attn_varlen needs a caller-provided device workspace (the longest-first
// work list and an error word).  Some callers have no way to provide one: a
// plugin that is handed only raw input/output pointers and no allocator, a
// serving host whose memory pool is sized once at start-up and forbids further
// device allocation, or a latency-critical loop that cannot afford the device
// synchronisation cudaMalloc may imply.  This entry point keeps that workspace
// in a fixed, file-scope device array instead, so the call allocates nothing.
//
// The array lives in every GPU's memory once the library is loaded there, until
// the process exits.  Host code must not pass the array's name to a kernel: on
// the host that name is only a stand-in for the symbol, not a device address.
// Its device address is looked up once per device with cudaGetSymbolAddress.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.cuh"
#include "vitfp8.h"

namespace {

constexpr int32_t kMaxSeqs = VITFP8_NOALLOC_MAX_SEQS;
// Same layout as a caller workspace: 64-byte header, one 16-byte record per
// segment, the key-range split's counters and partial results.
constexpr size_t kScratchBytes = vitfp8::ws_bytes(kMaxSeqs);

static __device__ __align__(256) uint8_t g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up on first use).
vitfp8_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VITFP8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return VITFP8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr)
            return VITFP8_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return VITFP8_OK;
}

}  // namespace

extern "C" vitfp8_status vitfp8_attn_varlen_noalloc(
    const uint8_t* q8, const uint8_t* k8, const uint8_t* v8t, const vitfp8_scale_state* d_state,
    const int32_t* d_cu_seqlens, int32_t num_seqs, int32_t max_seqlen, int32_t total_tokens,
    int32_t H, int32_t D, int32_t D_pad, float sm_scale, vitfp8_bf16* out, cudaStream_t stream) {
    if (num_seqs > kMaxSeqs) return VITFP8_ERR_UNSUPPORTED;
    if (num_seqs <= 0 || total_tokens <= 0) {
        // Nothing to launch (or an argument error): the checks of the
        // workspace entry point decide which, without touching the scratch.
        return vitfp8_attn_varlen(q8, k8, v8t, d_state, d_cu_seqlens, num_seqs, max_seqlen,
                                  total_tokens, H, D, D_pad, sm_scale, out, nullptr, 0, stream);
    }
    void* scratch = nullptr;
    vitfp8_status s = scratch_on_current_device(&scratch);
    if (s != VITFP8_OK) return s;
    if (vitfp8_attn_workspace_size(num_seqs) > kScratchBytes) return VITFP8_ERR_UNSUPPORTED;
    return vitfp8_attn_varlen(q8, k8, v8t, d_state, d_cu_seqlens, num_seqs, max_seqlen,
                              total_tokens, H, D, D_pad, sm_scale, out, scratch, kScratchBytes,
                              stream);
}
