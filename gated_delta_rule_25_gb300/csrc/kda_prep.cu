// Per-chunk factors of the chunkwise KDA forward, one CTA per (chunk, head).
//
// For a chunk of L <= 64 tokens of one sequence and head ("Autoresearch on Kimi
// Delta Attention", section THE MECHANISM: inside a block of tokens the work is
// matrix products; "NVIDIA Kernel Design Agents optimize Kimi Delta Attention",
// section 03: in-kernel L2 normalisation of q and k, the cumulative decay inside
// each 64-token chunk, the triangular inverse):
//   qh, kh   rows of q, k divided by sqrt(|x|^2 + eps)
//   Gamma_r  = g_1 + ... + g_r                  (per key channel, fp32)
//   A_ij     = beta_i sum_c kh_ic kh_jc exp(Gamma_ic - Gamma_jc)      j < i
//   P_ij     = sum_c qh_ic kh_jc exp(Gamma_ic - Gamma_jc)             j <= i
//   X        = (I + A)^-1   (unit lower triangular, forward substitution in fp32)
//   w        = X Diag(beta) (kh * exp(Gamma)),   u = X Diag(beta) v
// plus qh * exp(Gamma), (kh * exp(Gamma_L - Gamma))^T and exp(Gamma_L) for the
// state recurrence.  Every exponential is of a difference Gamma_i - Gamma_j with
// i >= j, or of Gamma itself, so it lies in (0, 1]: deep decays underflow to zero
// and never overflow (the page's section 03 describes kernels that overflowed).
// Rows past the end of the sequence are zero (k = v = beta = g = 0).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <typename TIn>
__device__ inline float load_in(const TIn* p);
template <>
__device__ inline float load_in<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <>
__device__ inline float load_in<float>(const float* p) {
    return *p;
}

template <int DK, int DV>
struct PrepSmem {
    static constexpr int DKP = DK + 1;  // padded rows: conflict-free column walks
    static constexpr int DVP = DV + 1;
    float qn[kChunk * DKP];
    float kn[kChunk * DKP];
    float G[kChunk * DKP];
    float vs[kChunk * DVP];
    float bs[kChunk];
    float A[kChunk * (kChunk + 1)];
    float X[kChunk * (kChunk + 1)];
};

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kThreads) prep_kernel(Dims d, const TIn* __restrict__ q,
                                                        const TIn* __restrict__ k,
                                                        const TIn* __restrict__ v,
                                                        const float* __restrict__ g,
                                                        const float* __restrict__ beta,
                                                        uint8_t* __restrict__ ws) {
    using Sm = PrepSmem<DK, DV>;
    constexpr int DKP = Sm::DKP, DVP = Sm::DVP, AP = kChunk + 1;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    WsLayout W(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= hdr->total_chunks) return;
    const int4 ch = reinterpret_cast<const int4*>(ws + W.chunks)[c];
    const long long row0 = ch.y;
    const int L = ch.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = d.H;

    // ---- load (masked rows are zero)
    for (int e = tid; e < kChunk * DK; e += kThreads) {
        int r = e / DK, cc = e % DK;
        float qv = 0.f, kv = 0.f, gv = 0.f;
        if (r < L) {
            size_t off = ((size_t)(row0 + r) * H + h) * DK + cc;
            qv = load_in<TIn>(q + off);
            kv = load_in<TIn>(k + off);
            gv = g[off];
        }
        sm.qn[r * DKP + cc] = qv;
        sm.kn[r * DKP + cc] = kv;
        sm.G[r * DKP + cc] = gv;
    }
    for (int e = tid; e < kChunk * DV; e += kThreads) {
        int r = e / DV, cc = e % DV;
        sm.vs[r * DVP + cc] = r < L ? load_in<TIn>(v + ((size_t)(row0 + r) * H + h) * DV + cc) : 0.f;
    }
    if (tid < kChunk) sm.bs[tid] = tid < L ? beta[(size_t)(row0 + tid) * H + h] : 0.f;
    __syncthreads();

    // ---- L2 normalisation (one warp per row)
    for (int r = warp; r < kChunk; r += kThreads / 32) {
        float sq = 0.f, sk = 0.f;
        for (int cc = lane; cc < DK; cc += 32) {
            float a = sm.qn[r * DKP + cc], b = sm.kn[r * DKP + cc];
            sq += a * a;
            sk += b * b;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
        }
        float iq = rsqrtf(sq + 1e-6f), ik = rsqrtf(sk + 1e-6f);
        for (int cc = lane; cc < DK; cc += 32) {
            sm.qn[r * DKP + cc] *= iq;
            sm.kn[r * DKP + cc] *= ik;
        }
    }
    // ---- cumulative gate per channel
    if (tid < DK) {
        float acc = 0.f;
        for (int r = 0; r < kChunk; ++r) {
            acc += sm.G[r * DKP + tid];
            sm.G[r * DKP + tid] = acc;
        }
    }
    __syncthreads();

    // ---- A (strictly lower) and P (lower incl. diagonal); warp per row i
    const size_t fb = W.factors + ((size_t)c * H + h) * W.factor_bytes;
    FactorLayout F(DK, DV);
    __nv_bfloat16* gP = reinterpret_cast<__nv_bfloat16*>(ws + fb + F.p);
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        for (int j = lane; j < kChunk; j += 32) {
            float a = 0.f, p = 0.f;
            if (j <= i) {
                for (int cc = 0; cc < DK; ++cc) {
                    float e = __expf(sm.G[i * DKP + cc] - sm.G[j * DKP + cc]);
                    float kj = sm.kn[j * DKP + cc] * e;
                    a += sm.kn[i * DKP + cc] * kj;
                    p += sm.qn[i * DKP + cc] * kj;
                }
            }
            sm.A[i * AP + j] = (j < i) ? a * sm.bs[i] : 0.f;
            gP[op_index(i, j, kChunk)] = __float2bfloat16(j <= i ? p : 0.f);
        }
    }
    __syncthreads();

    // ---- X = (I + A)^-1, thread j owns column j
    if (tid < kChunk) {
        const int j = tid;
        for (int i = 0; i < kChunk; ++i) {
            float x = (i == j) ? 1.f : 0.f;
            if (i > j) {
                for (int m = 0; m < i; ++m) x -= sm.A[i * AP + m] * sm.X[m * AP + j];
            }
            sm.X[i * AP + j] = x;
        }
    }
    // ---- QG, KT, GL (need qn, kn, G unchanged)
    __nv_bfloat16* gQG = reinterpret_cast<__nv_bfloat16*>(ws + fb + F.qg);
    __nv_bfloat16* gKT = reinterpret_cast<__nv_bfloat16*>(ws + fb + F.kt);
    float* gGL = reinterpret_cast<float*>(ws + fb + F.gl);
    for (int e = tid; e < kChunk * DK; e += kThreads) {
        int r = e / DK, cc = e % DK;
        float Gr = sm.G[r * DKP + cc], Gl = sm.G[(kChunk - 1) * DKP + cc];
        gQG[op_index(r, cc, kChunk)] = __float2bfloat16(sm.qn[r * DKP + cc] * __expf(Gr));
        gKT[op_index(cc, r, DK)] = __float2bfloat16(sm.kn[r * DKP + cc] * __expf(Gl - Gr));
    }
    if (tid < DK) gGL[tid] = __expf(sm.G[(kChunk - 1) * DKP + tid]);
    __syncthreads();
    // kn <- beta * kn * exp(Gamma);  vs <- beta * vs
    for (int e = tid; e < kChunk * DK; e += kThreads) {
        int r = e / DK, cc = e % DK;
        sm.kn[r * DKP + cc] *= sm.bs[r] * __expf(sm.G[r * DKP + cc]);
    }
    for (int e = tid; e < kChunk * DV; e += kThreads) {
        int r = e / DV, cc = e % DV;
        sm.vs[r * DVP + cc] *= sm.bs[r];
    }
    __syncthreads();

    // ---- w = X (beta kh exp(Gamma)), u = X (beta v)
    __nv_bfloat16* gW = reinterpret_cast<__nv_bfloat16*>(ws + fb + F.w);
    __nv_bfloat16* gU = reinterpret_cast<__nv_bfloat16*>(ws + fb + F.u0);
    for (int e = tid; e < kChunk * DK; e += kThreads) {
        int i = e / DK, cc = e % DK;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc += sm.X[i * AP + j] * sm.kn[j * DKP + cc];
        gW[op_index(i, cc, kChunk)] = __float2bfloat16(acc);
    }
    for (int e = tid; e < kChunk * DV; e += kThreads) {
        int i = e / DV, cc = e % DV;
        float acc = 0.f;
        for (int j = 0; j <= i; ++j) acc += sm.X[i * AP + j] * sm.vs[j * DVP + cc];
        gU[u0_index(i, cc)] = __float2bfloat16(acc);
    }
}

template <int DK, int DV, typename TIn>
cudaError_t launch_prep_t(const Dims& d, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, uint8_t* ws, cudaStream_t stream) {
    auto kern = prep_kernel<DK, DV, TIn>;
    size_t smem = sizeof(PrepSmem<DK, DV>);
    WsLayout W(d);
    if (W.cmax == 0) return cudaSuccess;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)W.cmax, (unsigned)d.H);
    kern<<<grid, kThreads, smem, stream>>>(d, static_cast<const TIn*>(q),
                                           static_cast<const TIn*>(k),
                                           static_cast<const TIn*>(v), g, beta, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep(const Dims& d, bool qkv_bf16, const void* q, const void* k,
                        const void* v, const float* g, const float* beta, uint8_t* ws,
                        cudaStream_t stream) {
#define KDA_PREP_CASE(DK_, DV_)                                                              \
    if (d.dk == DK_ && d.dv == DV_)                                                          \
        return qkv_bf16 ? launch_prep_t<DK_, DV_, __nv_bfloat16>(d, q, k, v, g, beta, ws, stream) \
                        : launch_prep_t<DK_, DV_, float>(d, q, k, v, g, beta, ws, stream);
    KDA_PREP_CASE(64, 64)
    KDA_PREP_CASE(64, 128)
    KDA_PREP_CASE(128, 64)
    KDA_PREP_CASE(128, 128)
#undef KDA_PREP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
