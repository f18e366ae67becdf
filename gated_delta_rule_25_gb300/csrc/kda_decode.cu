// One step of the KDA recurrence per sequence (single-token decode).
//
// For a sequence's state S (dk x dv, fp32) and its next token ("Autoresearch on
// Kimi Delta Attention", section THE MECHANISM: the per-token state update that
// the chunked form batches; "NVIDIA Kernel Design Agents optimize Kimi Delta
// Attention", section 03 REWARD HACKING: L2-normalised q and k, per-channel decay):
//   a = exp(g),  kh = k / |k|,  qh = q / |q|
//   r = (Diag(a) S)^T kh                       (length dv)
//   S' = Diag(a) S + beta kh (v - r)^T         = (I - beta kh kh^T) Diag(a) S + beta kh v^T
//   o = scale S'^T qh = scale ((Diag(a) S)^T qh + beta (qh . kh) (v - r))
// One pass over S gives both reductions, (Diag(a) S)^T kh and (Diag(a) S)^T qh; the
// update then rewrites S from the same registers.  The work is a read and a write
// of the state, so the kernel is bound by HBM bandwidth.
//
// One CTA per (sequence, head, 32-column value tile); 8 warps, warp w holds rows
// [w dk/8, (w+1) dk/8) of the tile, lane l column l, so every state access of a
// warp is one 128-byte line.
#include <cmath>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kDecThreads = 256, kDecWarps = 8, kDecCols = 32;

__device__ inline float to_f(float x) { return x; }
__device__ inline float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ inline void from_f(float& d, float x) { d = x; }
__device__ inline void from_f(__nv_bfloat16& d, float x) { d = __float2bfloat16(x); }

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta,
                  const float* h_in, float* h_out, float scale, T* __restrict__ o) {
    constexpr int RPW = DK / kDecWarps, NVT = DV / kDecCols, EPL = DK / 32;
    __shared__ float s_al[DK], s_ka[DK], s_qa[DK], s_kh[DK];
    __shared__ float s_red[kDecWarps][2][kDecCols];
    __shared__ float s_qk;
    const int nh = blockIdx.x / NVT, vt = blockIdx.x % NVT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = vt * kDecCols + lane;
    const size_t sbase = (size_t)nh * DK * DV;

    // the state tile first: its loads are in flight while the vectors are prepared
    float S[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
        S[r] = h_in ? h_in[sbase + (size_t)(warp * RPW + r) * DV + col] : 0.f;

    if (warp == 0) {
        float qv[EPL], kv[EPL], sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[e] = to_f(q[(size_t)nh * DK + lane * EPL + e]);
            kv[e] = to_f(k[(size_t)nh * DK + lane * EPL + e]);
            sq = fmaf(qv[e], qv[e], sq);
            sk = fmaf(kv[e], kv[e], sk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        const float iq = rsqrtf(sq + KDA_L2_EPS), ik = rsqrtf(sk + KDA_L2_EPS);
        float qk = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int i = lane * EPL + e;
            const float qh = qv[e] * iq, kh = kv[e] * ik, a = __expf(g[(size_t)nh * DK + i]);
            qk = fmaf(qh, kh, qk);
            s_al[i] = a;
            s_ka[i] = kh * a;
            s_qa[i] = qh * a;
            s_kh[i] = kh;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
        if (lane == 0) s_qk = qk;
    }
    __syncthreads();

    // partial reductions over this warp's rows
    float pr = 0.f, ps = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int i = warp * RPW + r;
        pr = fmaf(s_ka[i], S[r], pr);
        ps = fmaf(s_qa[i], S[r], ps);
    }
    s_red[warp][0][lane] = pr;
    s_red[warp][1][lane] = ps;
    __syncthreads();
    float rk = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) rk += s_red[w][0][lane];
    const float bt = beta[nh];
    const float u = to_f(v[(size_t)nh * DV + col]) - rk;  // v - (Diag(a) S)^T kh
    if (warp == 0) {
        float rq = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) rq += s_red[w][1][lane];
        from_f(o[(size_t)nh * DV + col], scale * fmaf(bt * s_qk, u, rq));
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int i = warp * RPW + r;
        h_out[sbase + (size_t)i * DV + col] = fmaf(s_al[i], S[r], bt * s_kh[i] * u);
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_decode_t(int NH, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h_in, float* h_out, float scale,
                            void* o, cudaStream_t stream) {
    const unsigned grid = (unsigned)NH * (DV / kDecCols);
    decode_kernel<DK, DV, T><<<grid, kDecThreads, 0, stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), g, beta,
        h_in, h_out, scale, static_cast<T*>(o));
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kda

extern "C" kda_status kda_decode(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                 const float* g, const float* beta, const float* h_in,
                                 float* h_out, int N, int H, int dk, int dv, float scale, void* o,
                                 kda_stream_t stream) {
    if (qkv_dtype != KDA_BF16 && qkv_dtype != KDA_FP32) return KDA_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || !std::isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return KDA_ERR_UNSUPPORTED;
    if ((long long)N * H > (1LL << 31) / 8) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !h_out || !o) return KDA_ERR_INVALID_ARG;
    using kda::aligned16;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(h_in) || !aligned16(h_out) || !aligned16(o))
        return KDA_ERR_ALIGNMENT;
    // h_out either is h_in or does not overlap it
    if (h_in && h_in != h_out) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(h_in), b0 = reinterpret_cast<uintptr_t>(h_out);
        const uintptr_t n = (uintptr_t)N * H * dk * dv * sizeof(float);
        if (a0 < b0 + n && b0 < a0 + n) return KDA_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int NH = N * H;
    const bool bf = qkv_dtype == KDA_BF16;
    cudaError_t e = cudaErrorInvalidValue;
#define KDA_DECODE_CASE(DK_, DV_)                                                                   \
    if (dk == DK_ && dv == DV_)                                                                     \
        e = bf ? kda::launch_decode_t<DK_, DV_, __nv_bfloat16>(NH, q, k, v, g, beta, h_in, h_out,    \
                                                                scale, o, s)                         \
               : kda::launch_decode_t<DK_, DV_, float>(NH, q, k, v, g, beta, h_in, h_out, scale, o, s);
    KDA_DECODE_CASE(64, 64)
    KDA_DECODE_CASE(64, 128)
    KDA_DECODE_CASE(128, 64)
    KDA_DECODE_CASE(128, 128)
#undef KDA_DECODE_CASE
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
