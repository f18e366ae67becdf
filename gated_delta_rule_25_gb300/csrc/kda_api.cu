// C ABI of the KDA prefill forward: argument checks, workspace carving, launches.
// Declarations and the contract are in include/kda.h.
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

cudaError_t ensure_smem_raw(const void* kern, size_t bytes) {
    static std::mutex mu;
    static std::map<const void*, uint64_t> done;  // kernel -> mask of devices set up
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    uint64_t& mask = done[kern];
    if (bit && (mask & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) mask |= bit;
    return e;
}

int num_sms() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    cache[dev] = n;
    return n;
}

}  // namespace kda

namespace {

std::atomic<int> g_pipeline{KDA_PIPELINE_AUTO};

// The fused pipeline's grid for these sizes under the current setting, or 0 for the
// split pipeline.  Automatic choice: where the fused pipeline was measured faster on
// GB300 (the throughput sweep of 22 shapes): fixed-length batches with B * H from 32
// to 256 whose split pipeline would run the tiled state kernel (B * H = 32 and 64:
// 6-16 %).  Where the split pipeline takes the 128-column chain kernel (B * H = 128
// and 256 at 128-chunk chains: 2-5 % faster split), for varlen batches (the chains of
// a round differ in length), B * H = 16 (its few chain CTAs bound it) and B * H >= 512
// (the factor CTAs it gives up cost more than the chains gain), the split one.
int pipeline_grid(const kda::Dims& d) {
    const int p = g_pipeline.load();
    if (p == KDA_PIPELINE_SPLIT || p == KDA_PIPELINE_SPLIT_WHOLE) return 0;
    const int grid = kda::fused_grid(d);
    if (grid == 0 || p == KDA_PIPELINE_FUSED) return grid;
    const long long pairs = (long long)d.N * d.H;
    const bool uniform = !d.varlen || d.N == 1;
    return uniform && pairs >= 32 && pairs <= 256 && !kda::chain128_pick_uniform(d) ? grid : 0;
}

bool valid_head_dim(int x) { return x == 64 || x == 128; }

// The split pipeline's state kernel: 0 tiled, 1 the 128-column chains, 2 decided on
// the device from the chain lengths (varlen batches of at least 512 chains; the
// 128-column kernel was never picked below that on the sweep's shapes, and the
// decision costs a launch of the kernel not chosen).
int c128_mode(const kda::Dims& d) {
    if (!kda::chain128_applies(d)) return 0;
    if (d.varlen && d.N > 1) return (long long)d.N * d.H >= 512 ? 2 : 0;
    return kda::chain128_pick_uniform(d) ? 1 : 0;
}

// Segmented chains (split pipeline, few long chains, a workspace with the segment
// region): the segment length for equal-length chains (0: none), or -1 for varlen
// batches long enough that segments may pay, decided on the device from the lengths
// (the tiled state kernel and the segment kernels are then all launched; those not
// chosen leave at once).
int seg_mode(const kda::Dims& d, size_t workspace_bytes) {
    if (g_pipeline.load() == KDA_PIPELINE_SPLIT_WHOLE) return 0;
    if (!kda::seg_layout_applies(d) || d.N > kda::kRankMax) return 0;
    if (workspace_bytes < kda::WsLayout(d).total_seg) return 0;
    if (!d.varlen || d.N == 1) return kda::seg_pick_uniform(d);
    return (long long)d.T >= 32LL * kda::kChunk ? -1 : 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks sizes; fills Dims.  Returns KDA_OK or the status to report.
kda_status make_dims(int B, int T, int H, int dk, int dv, int num_seqs, bool varlen,
                     kda::Dims& d) {
    if (B < 0 || T < 0 || H <= 0 || num_seqs < 0) return KDA_ERR_INVALID_ARG;
    if (!valid_head_dim(dk) || !valid_head_dim(dv)) return KDA_ERR_UNSUPPORTED;
    if (varlen) {
        if (B != 1) return KDA_ERR_INVALID_ARG;
    } else if (num_seqs != B) {
        return KDA_ERR_INVALID_ARG;
    }
    // token-head rows and grid sizes stay well inside 32-bit launch limits
    if ((long long)B * T * H > (1LL << 31) / 4) return KDA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H * 4 > (1LL << 31) - 1) return KDA_ERR_UNSUPPORTED;
    d = kda::Dims{B, T, H, dk, dv, num_seqs, varlen};
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_fwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs) {
    // B == 1 may be either layout; the varlen bound (T/64 + N chunks) covers both.
    kda::Dims d;
    if (make_dims(B, T, H, dk, dv, num_seqs, B == 1, d) != KDA_OK) return 0;
    return kda::WsLayout(d).total_seg;
}

int kda_fwd_launch_count(int B, int T, int H, int dk, int dv, int num_seqs) {
    // schedule, fused; or schedule, factors, then the state kernels (see fwd_impl)
    if (kda_fwd_uses_fused(B, T, H, dk, dv, num_seqs)) return 2;
    kda::Dims d;
    if (make_dims(B, T, H, dk, dv, num_seqs, B == 1 && num_seqs != B, d) != KDA_OK) return 3;
    const int seg = seg_mode(d, kda::WsLayout(d).total_seg);
    if (seg > 0) return 5;   // schedule, factors, pass A, scan, pass C
    if (seg < 0) return 6;   // ... and the tiled state kernel before the passes
    return c128_mode(d) == 2 ? 4 : 3;
}

void kda_set_pipeline(kda_pipeline pipeline) {
    g_pipeline.store(pipeline == KDA_PIPELINE_SPLIT          ? KDA_PIPELINE_SPLIT
                     : pipeline == KDA_PIPELINE_SPLIT_WHOLE ? KDA_PIPELINE_SPLIT_WHOLE
                     : pipeline == KDA_PIPELINE_FUSED       ? KDA_PIPELINE_FUSED
                                                            : KDA_PIPELINE_AUTO);
}

kda_pipeline kda_get_pipeline(void) { return static_cast<kda_pipeline>(g_pipeline.load()); }

int kda_fwd_uses_fused(int B, int T, int H, int dk, int dv, int num_seqs) {
    kda::Dims d;
    if (make_dims(B, T, H, dk, dv, num_seqs, B == 1 && num_seqs != B, d) != KDA_OK) return 0;
    return pipeline_grid(d) > 0 ? 1 : 0;
}

}  // extern "C"

namespace {

kda_status fwd_impl(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                    const void* g, kda_dtype g_dtype, const float* beta, const float* h0,
                    const int32_t* cu_seqlens, int num_seqs,
                    int B, int T, int H, int dk, int dv, float scale,
                    void* o, float* hT,
                    void* workspace, size_t workspace_bytes, kda_stream_t stream,
                    void* const* events) {
    if (qkv_dtype != KDA_BF16 && qkv_dtype != KDA_FP32) return KDA_ERR_UNSUPPORTED;
    if (g_dtype != KDA_FP32 && !(g_dtype == KDA_BF16 && qkv_dtype == KDA_BF16))
        return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    kda::Dims d;
    kda_status st = make_dims(B, T, H, dk, dv, num_seqs, cu_seqlens != nullptr, d);
    if (st != KDA_OK) return st;
    const bool any_tokens = (long long)B * T > 0;
    if (any_tokens && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o) ||
        !aligned16(beta) || !aligned16(h0) || !aligned16(hT) || !aligned16(cu_seqlens))
        return KDA_ERR_ALIGNMENT;
    kda::WsLayout W(d);
    if (!workspace || workspace_bytes < W.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KDA_ERR_WORKSPACE;
    if (num_seqs == 0) return KDA_OK;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool bf16 = qkv_dtype == KDA_BF16;
    int ev = 0;
    auto mark = [&]() -> bool {
        if (!events) return true;
        return cudaEventRecord(static_cast<cudaEvent_t>(events[ev++]), s) == cudaSuccess;
    };
    const bool gbf = g_dtype == KDA_BF16;
    const int grid = pipeline_grid(d);
    if (grid > 0) {
        if (!mark() || kda::launch_schedule_fused(d, cu_seqlens, ws, grid, kda::fused_ratio(d, bf16), s) !=
                           cudaSuccess)
            return KDA_ERR_CUDA;
        if (!mark()) return KDA_ERR_CUDA;
        const cudaError_t ce = kda::launch_fused(d, bf16, gbf, q, k, v, g, beta, h0, scale, o, hT, ws, s);
        if (ce != cudaSuccess || !mark()) return KDA_ERR_CUDA;
        return KDA_OK;
    }
    // split: the state recurrence on value tiles or, dk = dv = 128, on 128-column
    // chains where that is predicted faster (decided here for equal-length chains,
    // by the schedule kernel from the lengths for varlen batches, in which case both
    // kernels are launched and the one not chosen leaves at once)
    // (or, for few long chains, on segments: seg_mode)
    const int mode = c128_mode(d);
    const int seg = seg_mode(d, workspace_bytes);
    if (!mark() || kda::launch_schedule(d, cu_seqlens, ws, kda::split_nv_for(d), mode, seg, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (!mark() || kda::launch_prep_tc(d, bf16, gbf, q, k, v, g, beta, ws, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    cudaError_t ce;
    if (seg > 0) {
        if (!mark() || kda::launch_seg_pass(d, bf16, 0, h0, scale, o, hT, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark() || kda::launch_seg_scan(d, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark() || kda::launch_seg_pass(d, bf16, 1, h0, scale, o, hT, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark()) return KDA_ERR_CUDA;
        return KDA_OK;
    }
    if (mode != 1) {
        if (!mark()) return KDA_ERR_CUDA;
        ce = kda::launch_chain(d, bf16, h0, scale, o, hT, ws, s);
        if (ce != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (mode != 0) {
        if (!mark()) return KDA_ERR_CUDA;
        ce = kda::launch_chain128(d, bf16, h0, scale, o, hT, ws, s);
        if (ce != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (seg < 0) {
        if (!mark() || kda::launch_seg_pass(d, bf16, 0, h0, scale, o, hT, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark() || kda::launch_seg_scan(d, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (!mark() || kda::launch_seg_pass(d, bf16, 1, h0, scale, o, hT, ws, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (!mark()) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                   const float* g, const float* beta, const float* h0,
                   const int32_t* cu_seqlens, int num_seqs,
                   int B, int T, int H, int dk, int dv, float scale,
                   void* o, float* hT,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    return fwd_impl(q, k, v, qkv_dtype, g, KDA_FP32, beta, h0, cu_seqlens, num_seqs, B, T, H, dk,
                    dv, scale, o, hT, workspace, workspace_bytes, stream, nullptr);
}

kda_status kda_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                      const void* g, kda_dtype g_dtype, const float* beta, const float* h0,
                      const int32_t* cu_seqlens, int num_seqs,
                      int B, int T, int H, int dk, int dv, float scale,
                      void* o, float* hT,
                      void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    return fwd_impl(q, k, v, qkv_dtype, g, g_dtype, beta, h0, cu_seqlens, num_seqs, B, T, H, dk,
                    dv, scale, o, hT, workspace, workspace_bytes, stream, nullptr);
}

kda_status kda_fwd_profiled(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* beta, const float* h0,
                            const int32_t* cu_seqlens, int num_seqs,
                            int B, int T, int H, int dk, int dv, float scale,
                            void* o, float* hT,
                            void* workspace, size_t workspace_bytes, kda_stream_t stream,
                            void* const* events) {
    if (!events) return KDA_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, qkv_dtype, g, g_dtype, beta, h0, cu_seqlens, num_seqs, B, T, H, dk,
                    dv, scale, o, hT, workspace, workspace_bytes, stream, events);
}

kda_status kda_fwd_check(const void* workspace, kda_stream_t stream, uint32_t* device_error) {
    if (!workspace) return KDA_ERR_WORKSPACE;
    kda::Header hdr{};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&hdr, workspace, sizeof(hdr), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (device_error) *device_error = hdr.error;
    return hdr.error ? KDA_ERR_DEVICE : KDA_OK;
}

size_t kda_bwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs) {
    kda::Dims d;
    if (make_dims(B, T, H, dk, dv, num_seqs, B == 1, d) != KDA_OK) return 0;
    return kda::bwd_workspace_bytes(d);
}

kda_status kda_bwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                   const float* g, const float* beta, const float* h0,
                   const int32_t* cu_seqlens, int num_seqs,
                   int B, int T, int H, int dk, int dv, float scale,
                   const void* dout, const float* dhT,
                   float* dq, float* dk_out, float* dv_out, float* dg, float* dbeta, float* dh0,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    if (qkv_dtype != KDA_BF16 && qkv_dtype != KDA_FP32) return KDA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    kda::Dims d;
    kda_status st = make_dims(B, T, H, dk, dv, num_seqs, cu_seqlens != nullptr, d);
    if (st != KDA_OK) return st;
    const bool any_tokens = (long long)B * T > 0;
    if (any_tokens && (!q || !k || !v || !g || !beta || !dout || !dq || !dk_out || !dv_out || !dg || !dbeta))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(h0) || !aligned16(dout) || !aligned16(dhT) || !aligned16(dq) || !aligned16(dk_out) ||
        !aligned16(dv_out) || !aligned16(dg) || !aligned16(dbeta) || !aligned16(dh0) || !aligned16(cu_seqlens))
        return KDA_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < kda::bwd_workspace_bytes(d) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KDA_ERR_WORKSPACE;
    if (num_seqs == 0) return KDA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (kda::launch_schedule(d, cu_seqlens, ws, kda::kNV, 0, 0, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_bwd(d, qkv_dtype == KDA_BF16, cu_seqlens, q, k, v, g, beta, h0, dout, dhT, scale, dq,
                        dk_out, dv_out, dg, dbeta, dh0, ws, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

const char* kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported size or dtype";
        case KDA_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
        case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_DEVICE: return "device reported malformed input";
        case KDA_ERR_TOO_LARGE: return "problem too large for the built-in no-allocation scratch";
    }
    return "unknown status";
}

}  // extern "C"
