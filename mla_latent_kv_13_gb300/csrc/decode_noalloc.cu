// decode_noalloc.cu -- mla_decode_attention_noalloc: decode attention for callers that
// cannot hand the library a workspace.
//
// Some callers have no way to obtain device memory for scratch: code that runs while
// a stream is being captured into a CUDA graph (a cudaMalloc there is illegal or
// breaks the capture), plugins inside a host framework that owns every device
// allocation and exposes only tensor pointers, and serving loops that must not call
// cudaMalloc/cudaFree on their hot path because those calls can synchronise the
// device. For them, the scratch that the split-KV path needs (the per-range partial
// outputs, their log-sum-exps and the device error word) lives here, in one
// file-scope device array that is part of the loaded library image.
//
// The array occupies MLA_NOALLOC_SCRATCH_BYTES on every GPU that loads the library,
// until the process exits. Every call shares it and it keeps whatever the last call
// left there, so two calls that overlap on the GPU (different streams, or different
// host threads) corrupt each other's partial results: callers must serialise them.
#include "common.cuh"
#include "kernels.h"

#include <atomic>

namespace {

constexpr size_t kScratchBytes = MLA_NOALLOC_SCRATCH_BYTES;

// Device-side scratch: header (error word) | partial outputs | partial log-sum-exps.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];  // per-device address of the array

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array on the current device. The first call on a
// device resolves it (a query, not an allocation); later calls reuse it.
mla_status_t scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return MLA_ERR_CUDA;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_attention_noalloc(
    const mla_bf16_t *q_lat, const mla_bf16_t *q_rope, const mla_bf16_t *kv_cache,
    int num_blocks, const int32_t *block_table, int max_blocks, const int32_t *seqlens, int B,
    int H, int max_seqlen, float scale, int num_splits, mla_bf16_t *out, float *lse,
    mla_stream_t stream) {
    // The same argument checks as mla_decode_attention, then the scratch-size limit: a
    // rejected call returns before anything is queued on the device (the shared array's
    // header may belong to a call still running on another stream).
    mla_status_t st = mla::decode_validate(q_lat, q_rope, kv_cache, num_blocks, block_table,
                                           max_blocks, seqlens, B, 1, H, max_seqlen, scale,
                                           num_splits, out, lse);
    if (st != MLA_OK) return st;
    size_t need = 0;
    if ((st = mla_decode_workspace_size(B, H, max_seqlen, num_splits, &need)) != MLA_OK)
        return st;
    if (need > kScratchBytes) return MLA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_on_current_device(&scratch)) != MLA_OK) return st;
    // The error word must start at zero; the partial buffers are fully rewritten by
    // the attention kernel before the combine reads them.
    if (cudaMemsetAsync(scratch, 0, MLA_WS_HEADER_BYTES, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    return mla_decode_attention(q_lat, q_rope, kv_cache, num_blocks, block_table, max_blocks,
                                seqlens, B, H, max_seqlen, scale, num_splits, scratch,
                                round256(need), out, lse, stream);
}
