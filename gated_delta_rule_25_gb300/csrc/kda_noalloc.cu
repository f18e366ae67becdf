// kda_fwd_noalloc: the KDA forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory at the point where they run
// the forward: a plugin inside a host engine that owns every device allocation
// and hands out none, code on a path where an allocation's latency or possible
// failure is not acceptable, or a runtime whose allocator this library cannot
// reach.  For them this entry point takes only inputs and outputs: its scratch
// (the chunk schedule and the per-chunk factors that kda_fwd keeps in the
// caller's workspace) lives in one file-scope device array of a fixed size,
// KDA_NOALLOC_SCRATCH_BYTES.  Every GPU that loads this library holds that array
// until the process exits.
#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

// The built-in scratch.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) uint8_t g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v,
                                      kda_dtype qkv_dtype, const float* g, const float* beta,
                                      const float* h0, const int32_t* cu_seqlens, int num_seqs,
                                      int B, int T, int H, int dk, int dv, float scale, void* o,
                                      float* hT, kda_stream_t stream) {
    // Size check first: too-large problems are refused before any CUDA call.
    if (B < 0 || T < 0 || H <= 0 || num_seqs < 0) return KDA_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return KDA_ERR_UNSUPPORTED;
    if (cu_seqlens ? B != 1 : num_seqs != B) return KDA_ERR_INVALID_ARG;
    const kda::Dims d{B, T, H, dk, dv, num_seqs, cu_seqlens != nullptr};
    if (kda::WsLayout(d).total > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_TOO_LARGE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_fwd(q, k, v, qkv_dtype, g, beta, h0, cu_seqlens, num_seqs, B, T, H, dk, dv, scale,
                   o, hT, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" kda_status kda_fwd_noalloc_check(kda_stream_t stream, uint32_t* device_error) {
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    kda::Header hdr{};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&hdr, scratch, sizeof(hdr), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (device_error) *device_error = hdr.error;
    return hdr.error ? KDA_ERR_DEVICE : KDA_OK;
}
