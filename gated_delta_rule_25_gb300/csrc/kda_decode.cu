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
// One CTA per (sequence, head); 8 warps, warp w holds rows [w dk/8, (w+1) dk/8) of
// the state, each lane 4 consecutive value columns (16-byte accesses; a warp covers
// a whole row of dv = 128, or two rows of dv = 64).
#include <cmath>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kDecThreads = 256, kDecWarps = 8;

__device__ inline float to_f(float x) { return x; }
__device__ inline float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Four consecutive values as fp32, and back.
__device__ inline float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ inline float4 ld4(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ inline void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ inline void st4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(p) =
        make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}
__device__ inline float4 fma4(float a, float4 x, float4 y) {
    return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ inline float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ inline float4 shfl_xor4(float4 v, int m) {
    return make_float4(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m),
                       __shfl_xor_sync(0xffffffffu, v.z, m), __shfl_xor_sync(0xffffffffu, v.w, m));
}

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta,
                  const float* h_in, float* h_out, float scale, T* __restrict__ o) {
    constexpr int LPR = DV / 4;            // lanes per state row
    constexpr int RPP = 32 / LPR;          // rows per warp pass
    constexpr int RPW = DK / kDecWarps;    // rows per warp
    constexpr int NR = RPW / RPP;          // rows per thread
    constexpr int EPL = DK / 32;
    __shared__ float s_al[DK], s_ka[DK], s_qa[DK], s_kh[DK];
    __shared__ float4 s_red[kDecWarps][2][LPR];
    __shared__ float s_qk;
    const int nh = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = lane % LPR, rsub = lane / LPR;
    const size_t sbase = (size_t)nh * DK * DV;
    auto row_of = [&](int r) { return warp * RPW + r * RPP + rsub; };

    // the state first: its loads are in flight while the vectors are prepared
    float4 S[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r)
        S[r] = h_in ? ld4(h_in + sbase + (size_t)row_of(r) * DV + cl * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);

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

    // partial reductions over this thread's rows, then over the warp's row passes
    float4 pr = make_float4(0.f, 0.f, 0.f, 0.f), ps = pr;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int i = row_of(r);
        pr = fma4(s_ka[i], S[r], pr);
        ps = fma4(s_qa[i], S[r], ps);
    }
#pragma unroll
    for (int m = LPR; m < 32; m <<= 1) {
        pr = add4(pr, shfl_xor4(pr, m));
        ps = add4(ps, shfl_xor4(ps, m));
    }
    if (rsub == 0) {
        s_red[warp][0][cl] = pr;
        s_red[warp][1][cl] = ps;
    }
    __syncthreads();
    float4 rk = s_red[0][0][cl];
#pragma unroll
    for (int w = 1; w < kDecWarps; ++w) rk = add4(rk, s_red[w][0][cl]);
    const float bt = beta[nh];
    const float4 vv = ld4(v + (size_t)nh * DV + cl * 4);
    const float4 u = make_float4(vv.x - rk.x, vv.y - rk.y, vv.z - rk.z, vv.w - rk.w);  // v - (Diag(a) S)^T kh
    if (warp == 0 && rsub == 0) {
        float4 rq = s_red[0][1][cl];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) rq = add4(rq, s_red[w][1][cl]);
        const float c = bt * s_qk;
        st4(o + (size_t)nh * DV + cl * 4,
            make_float4(scale * fmaf(c, u.x, rq.x), scale * fmaf(c, u.y, rq.y),
                        scale * fmaf(c, u.z, rq.z), scale * fmaf(c, u.w, rq.w)));
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const int i = row_of(r);
        const float a = s_al[i], kb = bt * s_kh[i];
        st4(h_out + sbase + (size_t)i * DV + cl * 4,
            make_float4(fmaf(a, S[r].x, kb * u.x), fmaf(a, S[r].y, kb * u.y),
                        fmaf(a, S[r].z, kb * u.z), fmaf(a, S[r].w, kb * u.w)));
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_decode_t(int NH, const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h_in, float* h_out, float scale,
                            void* o, cudaStream_t stream) {
    const unsigned grid = (unsigned)NH;
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
