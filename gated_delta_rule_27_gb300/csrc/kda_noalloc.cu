// kda_noalloc.cu -- chunked prefill for callers that cannot allocate device
// memory.
//
// kda_prefill_chunked needs scratch ("workspace") from its caller.  Some
// callers have no way to provide it: code that runs while a stream is being
// captured, code inside a serving loop whose memory pool is sized up front and
// must never see a new cudaMalloc (which can also synchronise the device),
// and plugins whose host framework hands them only the input and output
// buffers.  kda_prefill_chunked_noalloc serves them: its scratch is one
// fixed-size array in the library's own device memory, so the call performs
// no allocation of any kind.
//
// The array lives in every GPU's memory from the moment the library's device
// code is loaded on that GPU until the process exits.  All calls on one GPU
// share it, so two calls whose kernels overlap on that GPU (different streams,
// no ordering between them) would corrupt each other; calls in one stream, or
// otherwise ordered, are safe.  Nothing in the array has to start at zero:
// every byte a call reads was written earlier in the same call.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr size_t kScratchBytes = KDA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Host code must not use this name as a device address:
// on the host it is only a stand-in that identifies the symbol.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and remembered.
kda_status scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_CUDA;
    if (dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return KDA_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v, const float *g,
                                       const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                                       int32_t chunk_size, const float *S0, void *o, float *S_final, void *stream) {
    const size_t need = kda_prefill_workspace_size(total_tokens, num_seqs, H, d_k, d_v, in_dtype, chunk_size);
    if (need == 0) {  // invalid or unsupported sizes: let the regular entry point name the error
        return kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                                   chunk_size, S0, o, S_final, nullptr, 0, stream);
    }
    if (need > kScratchBytes) return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const kda_status st = scratch_for_current_device(&scratch);
    if (st != KDA_OK) return st;
    return kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, H, d_k, d_v, in_dtype,
                               chunk_size, S0, o, S_final, scratch, kScratchBytes, stream);
}

kda_status kda_prefill_noalloc_check(void *stream) {
    void *scratch = nullptr;
    const kda_status st = scratch_for_current_device(&scratch);
    if (st != KDA_OK) return st;
    return kda_prefill_check(scratch, stream);
}

}  // extern "C"
