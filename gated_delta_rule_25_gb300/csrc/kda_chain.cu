// State recurrence across chunks on the tcgen05 tensor cores: one CTA per
// (sequence, head, 32-column value tile).  The state's value columns evolve
// independently, so each value tile is a chain of its own.
//
// For each chunk of the sequence, in order ("Autoresearch on Kimi Delta
// Attention", section THE MECHANISM: the state moves sequentially between blocks
// of tokens; "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section
// 01 RESULTS: the recurrent state must stay fp32, a bf16 state loses accuracy):
//   U  = u - w S                                   GEMM1  M=64,  N=32, K=dk
//   O  = scale ((qh * exp(Gamma)) S + P U)         GEMM3  M=64,  N=32, K=dk + 64
//   S <- Diag(exp(Gamma_L)) S + KT U               GEMM2  M=dk,  N=32, K=64
// S lives in fp32 registers of the epilogue warps (one key channel per thread);
// a bf16 copy of S and of U in shared memory are the B operands of the MMAs,
// which accumulate in fp32 in tensor memory.
//
// Warp roles (192 threads):
//   warps 0-3  epilogue: TMEM -> registers, U and S updates, output stores
//              (warp w reads TMEM lanes 32w..32w+31)
//   warp 4     MMA issue (one thread)
//   warp 5     bulk copies of the chunk factors (one thread), two stages deep
// Every wait is bounded; a time-out sets KDA_DEVERR_TIMEOUT in the workspace
// error word and the CTA drains and leaves.
#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

namespace {

constexpr int kEpiThreads = 128;
constexpr int kThreads = 192;
constexpr int NV = kNV;

template <int DK>
struct __align__(128) ChainStage {
    __nv_bfloat16 W[kChunk * DK];    // operand layout, 64 x DK
    __nv_bfloat16 QG[kChunk * DK];   // operand layout, 64 x DK
    __nv_bfloat16 KT[DK * kChunk];   // operand layout, DK x 64
    __nv_bfloat16 P[kChunk * kChunk];
    __nv_bfloat16 U0[kChunk * NV];   // row-major 64 x 32 slab of u
    float GL[DK];
};

template <int DK>
struct __align__(128) ChainSmem {
    ChainStage<DK> st[2];
    __nv_bfloat16 Sop[2][NV * DK];   // operand layout, NV x DK, two copies (B of GEMM1 / GEMM3a)
    __nv_bfloat16 Uop[NV * kChunk];  // operand layout, NV x 64 (B of GEMM2 / GEMM3b)
    uint64_t full[2], empty[2], d1, d2, d3[2], sready, uready, fin;
    uint32_t tmem_base;
    int abort;
};

// TMEM columns: D1 [0, 32), D2 [32, 64), D3 double buffer [64, 128).
constexpr uint32_t kColD1 = 0, kColD2 = 32, kColD3 = 64, kTmemCols = 128;

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

// Row of an M-row accumulator held by (warp w, lane l) of the epilogue, or -1.
// M = 128: lane quarter w holds rows 32w..32w+31.  M = 64: lanes 0-15 of each
// quarter hold rows 16w..16w+15.
template <int M>
__device__ inline int acc_row(int w, int l) {
    if (M == 128) return 32 * w + l;
    return l < 16 ? 16 * w + l : -1;
}

__device__ inline void raise_error(uint8_t* ws, volatile int* abort) {
    *abort = 1;
    atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
}

template <int DK, int DV, typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
    chain_tc_kernel(Dims d, const float* __restrict__ h0, float scale, TOut* __restrict__ o,
                    float* __restrict__ hT, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ChainSmem<DK>& sm = *reinterpret_cast<ChainSmem<DK>*>(smem_raw);
    constexpr int NVT = DV / NV;
    const int vt = blockIdx.x % NVT;
    const int h = (blockIdx.x / NVT) % d.H;
    const int s = blockIdx.x / (NVT * d.H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WsLayout W(d);
    const FactorLayout F(DK, DV);
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int4* chunks = reinterpret_cast<const int4*>(ws + W.chunks);
    const int c0 = seq_first[s];
    const int nch = seq_first[s + 1] - c0;
    volatile int* abort = &sm.abort;

    if (tid == 0) {
        ptx::mbar_init(&sm.full[0], 1);
        ptx::mbar_init(&sm.full[1], 1);
        ptx::mbar_init(&sm.empty[0], 1 + 4);
        ptx::mbar_init(&sm.empty[1], 1 + 4);
        ptx::mbar_init(&sm.d1, 1);
        ptx::mbar_init(&sm.d2, 1);
        ptx::mbar_init(&sm.d3[0], 1);
        ptx::mbar_init(&sm.d3[1], 1);
        ptx::mbar_init(&sm.sready, kEpiThreads);
        ptx::mbar_init(&sm.uready, kEpiThreads);
        ptx::mbar_init(&sm.fin, 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 5) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t main_bytes = (uint32_t)(F.u0 - F.w);  // W, QG, KT, P back to back
            const uint32_t u_bytes = kChunk * NV * 2, gl_bytes = DK * 4;
            int issued = 0;
            for (int j = 0; j < nch; ++j) {
                const int st = j & 1;
                if (j >= 2 && !ptx::mbar_wait_or_abort(&sm.empty[st], ((j >> 1) - 1) & 1, abort)) {
                    raise_error(ws, abort);
                    break;
                }
                const uint8_t* fb = ws + W.factors + ((size_t)(c0 + j) * d.H + h) * W.factor_bytes;
                ptx::mbar_arrive_expect_tx(&sm.full[st], main_bytes + u_bytes + gl_bytes);
                ptx::bulk_g2s(sm.st[st].W, fb + F.w, main_bytes, &sm.full[st]);
                ptx::bulk_g2s(sm.st[st].U0, fb + F.u0 + (size_t)vt * u_bytes, u_bytes, &sm.full[st]);
                ptx::bulk_g2s(sm.st[st].GL, fb + F.gl, gl_bytes, &sm.full[st]);
                issued = j + 1;
            }
            if (*abort) {  // let copies already in flight land before the CTA leaves
                volatile int never = 0;
                for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j)
                    ptx::mbar_wait_or_abort(&sm.full[j & 1], (j >> 1) & 1, &never);
            }
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t sop0 = ptx::smem_u32(sm.Sop[0]), uop = ptx::smem_u32(sm.Uop);
            constexpr uint32_t id_w = ptx::idesc_bf16(64, NV);
            constexpr uint32_t id_k = ptx::idesc_bf16(DK, NV);
            bool ok = true;
            for (int j = 0; j < nch && ok; ++j) {
                const int st = j & 1;
                ok = ptx::mbar_wait_or_abort(&sm.full[st], (j >> 1) & 1, abort) &&
                     ptx::mbar_wait_or_abort(&sm.sready, j & 1, abort);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t wa = ptx::smem_u32(sm.st[st].W), qa = ptx::smem_u32(sm.st[st].QG);
                const uint32_t ka = ptx::smem_u32(sm.st[st].KT), pa = ptx::smem_u32(sm.st[st].P);
                const uint32_t d3 = tmem + kColD3 + (uint32_t)(j & 1) * NV;
                const uint32_t sop = sop0 + (uint32_t)(j & 1) * (NV * DK * 2);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk)  // D1 = W S
                    ptx::mma_bf16(tmem + kColD1, ptx::smem_desc(wa + kk * 2048, 1024, 128),
                                  ptx::smem_desc(sop + kk * 2 * (NV / 8) * 128, (NV / 8) * 128, 128),
                                  id_w, kk > 0);
                ptx::mma_commit(&sm.d1);
                ok = ptx::mbar_wait_or_abort(&sm.uready, j & 1, abort);
                if (!ok) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)  // D2 = KT U (the serial path)
                    ptx::mma_bf16(tmem + kColD2,
                                  ptx::smem_desc(ka + kk * 2 * (DK / 8) * 128, (DK / 8) * 128, 128),
                                  ptx::smem_desc(uop + kk * 2 * (NV / 8) * 128, (NV / 8) * 128, 128),
                                  id_k, kk > 0);
                ptx::mma_commit(&sm.d2);
                // the output products are off the serial path: issued after D2.  They
                // read S copy j & 1; the epilogue writes the next state into the other
                // copy, and reuses this one only after d2 of chunk j + 1, whose commit
                // covers these MMAs.
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk)  // D3 = QG S
                    ptx::mma_bf16(d3, ptx::smem_desc(qa + kk * 2048, 1024, 128),
                                  ptx::smem_desc(sop + kk * 2 * (NV / 8) * 128, (NV / 8) * 128, 128),
                                  id_w, kk > 0);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)  // D3 += P U
                    ptx::mma_bf16(d3, ptx::smem_desc(pa + kk * 2048, 1024, 128),
                                  ptx::smem_desc(uop + kk * 2 * (NV / 8) * 128, (NV / 8) * 128, 128),
                                  id_w, true);
                ptx::mma_commit(&sm.d3[j & 1]);
                ptx::mma_commit(&sm.empty[st]);
            }
            if (!ok) raise_error(ws, abort);
            // all issued MMAs complete before TMEM is released
            ptx::mma_commit(&sm.fin);
            volatile int never = 0;
            ptx::mbar_wait_or_abort(&sm.fin, 0, &never);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int w = warp, l = lane;
        const uint32_t lane_base = (uint32_t)(32 * w) << 16;
        const int ch = acc_row<DK>(w, l);     // key channel of this thread's state row
        const int ur = acc_row<64>(w, l);     // chunk row of this thread in D1 / D3
        float S[NV];
        const size_t srow = ((size_t)s * d.H + h) * DK;
        if (ch >= 0) {
#pragma unroll
            for (int n = 0; n < NV; ++n)
                S[n] = h0 ? h0[(srow + ch) * DV + vt * NV + n] : 0.f;
#pragma unroll
            for (int n = 0; n < NV; ++n) sm.Sop[0][op_index(n, ch, NV)] = __float2bfloat16(S[n]);
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(&sm.sready);
        bool ok = true;
        for (int j = 0; j < nch; ++j) {
            const int st = j & 1;
            const int4 chk = chunks[c0 + j];
            float acc[NV];
            // (a) U = u - W S
            ok = ptx::mbar_wait_or_abort(&sm.d1, j & 1, abort) &&
                 ptx::mbar_wait_or_abort(&sm.full[st], (j >> 1) & 1, abort);
            if (!ok) break;
            ptx::tc_fence_after();
            ptx::tmem_ld16(tmem + lane_base + kColD1, *reinterpret_cast<float(*)[16]>(&acc[0]));
            ptx::tmem_ld16(tmem + lane_base + kColD1 + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
            ptx::tmem_ld_wait();
            if (ur >= 0) {
                const __nv_bfloat16* u0 = sm.st[st].U0 + ur * NV;
#pragma unroll
                for (int n = 0; n < NV; ++n)
                    sm.Uop[op_index(n, ur, NV)] = __float2bfloat16(__bfloat162float(u0[n]) - acc[n]);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.uready);
            // (b) S <- GL * S + KT U
            ok = ptx::mbar_wait_or_abort(&sm.d2, j & 1, abort);
            if (!ok) break;
            ptx::tc_fence_after();
            ptx::tmem_ld16(tmem + lane_base + kColD2, *reinterpret_cast<float(*)[16]>(&acc[0]));
            ptx::tmem_ld16(tmem + lane_base + kColD2 + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
            ptx::tmem_ld_wait();
            if (ch >= 0) {
                const float gl = sm.st[st].GL[ch];
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    S[n] = fmaf(gl, S[n], acc[n]);
                    sm.Sop[(j + 1) & 1][op_index(n, ch, NV)] = __float2bfloat16(S[n]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&sm.sready);
            __syncwarp();
            if (l == 0) ptx::mbar_arrive(&sm.empty[st]);
            // (c) O = scale * D3
            ok = ptx::mbar_wait_or_abort(&sm.d3[j & 1], (j >> 1) & 1, abort);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t d3 = tmem + lane_base + kColD3 + (uint32_t)(j & 1) * NV;
            ptx::tmem_ld16(d3, *reinterpret_cast<float(*)[16]>(&acc[0]));
            ptx::tmem_ld16(d3 + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            if (ur >= 0 && ur < chk.z) {
                TOut* orow = o + ((size_t)(chk.y + ur) * d.H + h) * DV + vt * NV;
#pragma unroll
                for (int n = 0; n < NV; ++n) store_out<TOut>(orow + n, scale * acc[n]);
            }
        }
        if (!ok) raise_error(ws, abort);
        if (hT && ch >= 0) {
#pragma unroll
            for (int n = 0; n < NV; ++n) hT[(srow + ch) * DV + vt * NV + n] = S[n];
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int DK, int DV, typename TOut>
cudaError_t launch_t(const Dims& d, const float* h0, float scale, void* o, float* hT, uint8_t* ws,
                     cudaStream_t stream) {
    auto kern = chain_tc_kernel<DK, DV, TOut>;
    const size_t smem = sizeof(ChainSmem<DK>);
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)d.N * d.H * (DV / NV);
    if (grid == 0) return cudaSuccess;
    kern<<<grid, kThreads, smem, stream>>>(d, h0, scale, static_cast<TOut*>(o), hT, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain(const Dims& d, bool qkv_bf16, const float* h0, float scale, void* o,
                         float* hT, uint8_t* ws, cudaStream_t stream) {
#define KDA_CHAIN_CASE(DK_, DV_)                                                             \
    if (d.dk == DK_ && d.dv == DV_)                                                          \
        return qkv_bf16 ? launch_t<DK_, DV_, __nv_bfloat16>(d, h0, scale, o, hT, ws, stream) \
                        : launch_t<DK_, DV_, float>(d, h0, scale, o, hT, ws, stream);
    KDA_CHAIN_CASE(64, 64)
    KDA_CHAIN_CASE(64, 128)
    KDA_CHAIN_CASE(128, 64)
    KDA_CHAIN_CASE(128, 128)
#undef KDA_CHAIN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
