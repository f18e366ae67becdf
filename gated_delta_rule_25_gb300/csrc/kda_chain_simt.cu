// State recurrence across chunks, plain fp32 CUDA-core version: one CTA per
// (sequence, head, 32-column value tile).  The state's value columns evolve
// independently, so a value tile is a chain of its own.
//
// For each chunk of the sequence, in order ("Autoresearch on Kimi Delta
// Attention", section THE MECHANISM: the state moves sequentially between blocks;
// "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 01: the
// recurrent state is kept in fp32, never bf16):
//   U  = u - w S                       (the corrections the chunk writes)
//   O  = scale ((qh * exp(Gamma)) S + P U)
//   S <- Diag(exp(Gamma_L)) S + (kh * exp(Gamma_L - Gamma))^T U
// This version serves as a cross-check of the tensor-core chain.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;
constexpr int NV = kNV;

template <int DK>
struct ChainSmem {
    float S[DK * NV];
    float Wm[kChunk * (DK + 1)];
    float QG[kChunk * (DK + 1)];
    float KT[DK * (kChunk + 1)];
    float P[kChunk * (kChunk + 1)];
    float U[kChunk * NV];
    float GL[DK];
};

template <typename TOut>
__device__ inline void store_out(TOut* p, float x);
template <>
__device__ inline void store_out<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16(x);
}
template <>
__device__ inline void store_out<float>(float* p, float x) {
    *p = x;
}

template <int DK, int DV, typename TOut>
__global__ void __launch_bounds__(kThreads) chain_simt_kernel(Dims d, const float* __restrict__ h0,
                                                              float scale, TOut* __restrict__ o,
                                                              float* __restrict__ hT,
                                                              const uint8_t* __restrict__ ws) {
    constexpr int DKP = DK + 1, CP = kChunk + 1;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ChainSmem<DK>& sm = *reinterpret_cast<ChainSmem<DK>*>(smem_raw);
    constexpr int NVT = DV / NV;
    const int vt = blockIdx.x % NVT;
    const int h = (blockIdx.x / NVT) % d.H;
    const int s = reinterpret_cast<const int32_t*>(ws + WsLayout(d).order)[blockIdx.x / (NVT * d.H)];
    const int tid = threadIdx.x, n = tid % NV, r8 = tid / NV;
    WsLayout W(d);
    FactorLayout F(DK, DV);
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int4* chunks = reinterpret_cast<const int4*>(ws + W.chunks);
    const int c0 = seq_first[s], c1 = seq_first[s + 1];

    for (int e = tid; e < DK * NV; e += kThreads) {
        int r = e / NV, cc = e % NV;
        sm.S[e] = h0 ? h0[(((size_t)s * d.H + h) * DK + r) * DV + vt * NV + cc] : 0.f;
    }
    for (int c = c0; c < c1; ++c) {
        const int4 ch = chunks[c];
        const uint8_t* fb = ws + W.factors + ((size_t)c * d.H + h) * W.factor_bytes;
        const __nv_bfloat16* gW = reinterpret_cast<const __nv_bfloat16*>(fb + F.w);
        const __nv_bfloat16* gQ = reinterpret_cast<const __nv_bfloat16*>(fb + F.qg);
        const __nv_bfloat16* gK = reinterpret_cast<const __nv_bfloat16*>(fb + F.kt);
        const __nv_bfloat16* gP = reinterpret_cast<const __nv_bfloat16*>(fb + F.p);
        const __nv_bfloat16* gU = reinterpret_cast<const __nv_bfloat16*>(fb + F.u0);
        const float* gGL = reinterpret_cast<const float*>(fb + F.gl);
        __syncthreads();  // previous chunk done with the tiles
        for (int e = tid; e < kChunk * DK; e += kThreads) {
            int r = e / DK, cc = e % DK;
            sm.Wm[r * DKP + cc] = __bfloat162float(gW[op_index(r, cc, kChunk)]);
            sm.QG[r * DKP + cc] = __bfloat162float(gQ[op_index(r, cc, kChunk)]);
            sm.KT[cc * CP + r] = __bfloat162float(gK[op_index(cc, r, DK)]);
        }
        for (int e = tid; e < kChunk * kChunk; e += kThreads) {
            int r = e / kChunk, j = e % kChunk;
            sm.P[r * CP + j] = __bfloat162float(gP[op_index(r, j, kChunk)]);
        }
        if (tid < DK) sm.GL[tid] = gGL[tid];
        __syncthreads();
        // U = u - w S
        for (int i = r8; i < kChunk; i += kThreads / NV) {
            float acc = __bfloat162float(gU[u0_index(i, vt * NV + n)]);
            for (int cc = 0; cc < DK; ++cc) acc -= sm.Wm[i * DKP + cc] * sm.S[cc * NV + n];
            sm.U[i * NV + n] = acc;
        }
        __syncthreads();
        // O = scale (QG S + P U)
        const int L = ch.z;
        const long long row0 = ch.y;
        for (int i = r8; i < L; i += kThreads / NV) {
            float acc = 0.f;
            for (int cc = 0; cc < DK; ++cc) acc += sm.QG[i * DKP + cc] * sm.S[cc * NV + n];
            for (int j = 0; j <= i; ++j) acc += sm.P[i * CP + j] * sm.U[j * NV + n];
            store_out<TOut>(o + ((size_t)(row0 + i) * d.H + h) * DV + vt * NV + n, scale * acc);
        }
        __syncthreads();
        // S <- GL * S + KT U
        for (int r = r8; r < DK; r += kThreads / NV) {
            float acc = sm.GL[r] * sm.S[r * NV + n];
            for (int j = 0; j < kChunk; ++j) acc += sm.KT[r * CP + j] * sm.U[j * NV + n];
            sm.S[r * NV + n] = acc;
        }
    }
    __syncthreads();
    if (hT) {
        for (int e = tid; e < DK * NV; e += kThreads) {
            int r = e / NV, cc = e % NV;
            hT[(((size_t)s * d.H + h) * DK + r) * DV + vt * NV + cc] = sm.S[e];
        }
    }
}

template <int DK, int DV, typename TOut>
cudaError_t launch_chain_t(const Dims& d, const float* h0, float scale, void* o, float* hT,
                           uint8_t* ws, cudaStream_t stream) {
    auto kern = chain_simt_kernel<DK, DV, TOut>;
    size_t smem = sizeof(ChainSmem<DK>);
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    unsigned grid = (unsigned)d.N * d.H * (DV / NV);
    if (grid == 0) return cudaSuccess;
    kern<<<grid, kThreads, smem, stream>>>(d, h0, scale, static_cast<TOut*>(o), hT, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain_simt(const Dims& d, bool qkv_bf16, const float* h0, float scale,
                              void* o, float* hT, uint8_t* ws, cudaStream_t stream) {
#define KDA_CHAIN_CASE(DK_, DV_)                                                           \
    if (d.dk == DK_ && d.dv == DV_)                                                        \
        return qkv_bf16 ? launch_chain_t<DK_, DV_, __nv_bfloat16>(d, h0, scale, o, hT, ws, stream) \
                        : launch_chain_t<DK_, DV_, float>(d, h0, scale, o, hT, ws, stream);
    KDA_CHAIN_CASE(64, 64)
    KDA_CHAIN_CASE(64, 128)
    KDA_CHAIN_CASE(128, 64)
    KDA_CHAIN_CASE(128, 128)
#undef KDA_CHAIN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
