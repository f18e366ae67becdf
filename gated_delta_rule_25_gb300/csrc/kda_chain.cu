// State recurrence across chunks on the tcgen05 tensor cores: one chain per
// (sequence, head, NV-column value tile), NV = 16, 32 or 64.  The state's value
// columns evolve independently, so each value tile is a chain of its own: 64-column
// tiles halve the number of chains (and the MMA issues per unit of work) when there
// are more chains than SMs, 16-column tiles put twice as many SMs to work when there
// are few.
//
// For each chunk of the sequence, in order ("Autoresearch on Kimi Delta
// Attention", section THE MECHANISM: the state moves sequentially between blocks
// of tokens; "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section
// 01 RESULTS: the recurrent state must stay fp32, a bf16 state loses accuracy):
//   [w S ; QG S]  = [w ; QG] S                     GEMM1  M=128, N=NV, K=dk
//   U  = u - w S
//   S <- Diag(exp(Gamma_L)) S + KT U               GEMM2  M=dk,  N=NV, K=64 (tf32)
//   O  = scale (QG S + P U)                        GEMM3  M=128, N=NV, K=64
// (QG = qh * exp(Gamma)).  w and QG arrive as one 128-row operand tile, so one
// product gives both w S (accumulator rows 0-63) and QG S (rows 64-127).  GEMM3
// accumulates P U onto rows 64-127 of the same accumulator: its A descriptor
// starts one 8-row block-row group (1 KB) before the 64-row P tile, so that rows
// 64-127 of the 128-row operand are exactly P (rows 0-63, already consumed, pick
// up a dead sum).  S lives in fp32 registers of the four epilogue warps (one key
// channel per thread).  bf16 copies of S and U in shared memory (N-major) are the
// B operands of GEMM1 and GEMM3; GEMM2, whose rounding would stay in the state,
// takes KT, u and U in fp32 (tf32 products).  All accumulate in fp32 in tensor
// memory.
//
// Only GEMM1 and GEMM2 are on the serial path.  Per chunk: thread 0 issues GEMM1;
// warps 0-1 form U from its rows 0-63 while warps 2-3 store the previous chunk's
// output (rows 64-127 of the other accumulator buffer); a named barrier; thread 0
// issues GEMM2 (and signals warp 5, which issues GEMM3), S is updated from D2, a
// named barrier, and the next chunk starts.
//
// The kernel is persistent (one CTA per SM): the producer warp takes work items
// (sequence, head, value tile), longest sequences first, from a counter in the
// workspace, streams each item's chunks through the stage ring and stamps every
// stage with its item; the other warps follow the stamps (a new item loads h0 at
// its first chunk and stores h_T after its last), so chains run back to back.
//
// Warps 0-3: epilogue, GEMM1/GEMM2 issue (warp w reads TMEM lanes 32w..32w+31).
// Warp 4: work items and bulk copies of the per-chunk factors, two stages deep.
// Warp 5: GEMM3 issue (output products, off the serial path).
// Every wait is bounded; a time-out sets KDA_DEVERR_TIMEOUT in the workspace
// error word and the CTA drains and leaves.
#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kAMajorMN = 1u << 15;  // instruction-descriptor bit: A is M-major
constexpr uint32_t kBMajorMN = 1u << 16;  // instruction-descriptor bit: B is N-major

// GEMM2's B operand: U^T (NV value columns x 64 chunk rows) in fp32, K-major core
// matrices of 8 columns x 4 rows (16 bytes each).  K-adjacent core matrices sit
// kU32Lbo = 144 bytes apart (not 128), so a warp's 32 consecutive chunk rows of one
// column hit 32 different banks when the epilogue writes them.
constexpr uint32_t kU32Lbo = 144, kU32Sbo = (kChunk / 4) * kU32Lbo;
template <int NV>
constexpr int u32_words() { return (NV / 8) * kU32Sbo / 4; }
__device__ inline int u32_index(int n, int r) {
    return (int)(((n >> 3) * kU32Sbo + (r >> 2) * kU32Lbo) / 4) + ((n & 7) << 2) + (r & 3);
}

template <int DK, int NV>
struct __align__(128) ChainStage {
    __nv_bfloat16 WQ[2 * kChunk * DK];  // M-major operand, 128 x DK: w, then QG
    float KT[DK * kChunk];           // tf32 operand layout, DK x 64
    __nv_bfloat16 P[kChunk * kChunk];
    float U0[kChunk * NV];           // NV/32 slabs of u, each [8 column groups][64 rows][4]
    float GL[DK];
    int4 item;                       // {sequence, head, value tile, chunk index j}
    int4 info;                       // {chunks of the item, first token row, rows, end marker}
};

template <int DK, int NV>
struct __align__(128) ChainSmem {
    ChainStage<DK, NV> st[kStages];
    __nv_bfloat16 Sop[NV * DK];      // N-major operand (B of GEMM1)
    __nv_bfloat16 Uop[NV * kChunk];  // N-major operand (B of GEMM3)
    float Uop32[u32_words<NV>()];    // K-major tf32 operand (B of GEMM2), padded
    uint64_t full[kStages], empty[kStages], d1, d2, d3[2], uready, fin, fin3;
    uint32_t tmem_base;
    int abort;
};

// TMEM columns: D1 (GEMM1, then GEMM3 on top) double buffer [0, 2 NV), D2 [2 NV, 3 NV).
template <int NV>
struct Cols {
    static constexpr uint32_t D1 = 0, D2 = 2 * NV, total = NV == 16 ? 64 : (NV == 32 ? 128 : 256);
};

// Element index of (n, k) in an N-major, unswizzled operand with N = NV rows:
// 8 x 8 core matrices, 8 consecutive n contiguous, n-blocks fastest.
template <int NV>
__device__ inline int nmaj_index(int n, int k) {
    return (((k >> 3) * (NV / 8) + (n >> 3)) << 6) + ((k & 7) << 3) + (n & 7);
}

__device__ inline uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Row of an M-row accumulator held by (warp w, lane l) of the epilogue, or -1.
// M = 128: lane quarter w holds rows 32w..32w+31.  M = 64: lanes 0-15 of each
// quarter hold rows 16w..16w+15.
template <int M>
__device__ inline int acc_row(int w, int l) {
    if (M == 128) return 32 * w + l;
    return l < 16 ? 16 * w + l : -1;
}

// Named barrier of the 128 epilogue threads that also ANDs a flag across them.
__device__ inline bool epi_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ inline void raise_error(uint8_t* ws, volatile int* abort) {
    *abort = 1;
    atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
}

// Writes NV output values of one row (bf16 or fp32) with 16-byte stores.
template <int NV>
__device__ inline void store_row(__nv_bfloat16* p, const float (&x)[NV], float scale) {
#pragma unroll
    for (int i = 0; i < NV; i += 8) {
        uint4 u = make_uint4(pack_bf16(scale * x[i], scale * x[i + 1]),
                             pack_bf16(scale * x[i + 2], scale * x[i + 3]),
                             pack_bf16(scale * x[i + 4], scale * x[i + 5]),
                             pack_bf16(scale * x[i + 6], scale * x[i + 7]));
        *reinterpret_cast<uint4*>(p + i) = u;
    }
}
template <int NV>
__device__ inline void store_row(float* p, const float (&x)[NV], float scale) {
#pragma unroll
    for (int i = 0; i < NV; i += 4)
        *reinterpret_cast<float4*>(p + i) =
            make_float4(scale * x[i], scale * x[i + 1], scale * x[i + 2], scale * x[i + 3]);
}

// NV consecutive TMEM columns of this warp's 32 lanes, then one wait.
template <int NV>
__device__ inline void tmem_ldnv(uint32_t taddr, float (&x)[NV]) {
#pragma unroll
    for (int i = 0; i < NV / 16; ++i)
        ptx::tmem_ld16(taddr + 16 * i, *reinterpret_cast<float(*)[16]>(&x[16 * i]));
    ptx::tmem_ld_wait();
}

template <int DK, int DV, int NV, typename TOut>
__global__ void __launch_bounds__(kThreads, 1)
    chain_tc_kernel(Dims d, const float* __restrict__ h0, float scale, TOut* __restrict__ o,
                    float* __restrict__ hT, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ChainSmem<DK, NV>& sm = *reinterpret_cast<ChainSmem<DK, NV>*>(smem_raw);
    constexpr uint32_t kColD1 = Cols<NV>::D1, kColD2 = Cols<NV>::D2, kTmemCols = Cols<NV>::total;
    constexpr int NVT = DV / NV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WsLayout W(d);
    const FactorLayout F(DK, DV);
    Header* hdr = reinterpret_cast<Header*>(ws + W.header);
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int32_t* order = reinterpret_cast<const int32_t*>(ws + W.order);
    const int4* chunks = reinterpret_cast<const int4*>(ws + W.chunks);
    const int n_items = d.N * d.H * NVT;
    volatile int* abort = &sm.abort;
    if (hdr->chain128 || hdr->seg) return;  // the 128-column or segmented chains run it instead

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            ptx::mbar_init(&sm.full[i], 1);
            ptx::mbar_init(&sm.empty[i], 3);  // two MMA commits + epilogue release
        }
        ptx::mbar_init(&sm.d1, 1);
        ptx::mbar_init(&sm.d2, 1);
        ptx::mbar_init(&sm.d3[0], 1);
        ptx::mbar_init(&sm.d3[1], 1);
        ptx::mbar_init(&sm.uready, 1);
        ptx::mbar_init(&sm.fin, 1);
        ptx::mbar_init(&sm.fin3, 1);
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

    if (warp == 4) {
        // ------------------------------------------------ work items + producer
        const uint32_t main_bytes = (uint32_t)(F.u0 - F.wq);  // WQ, KT, P back to back
        const uint32_t u_bytes = kChunk * NV * 4, gl_bytes = DK * 4;
        int gj = 0;
        bool okp = true;
        while (okp) {
            int item = 0;
            if (lane == 0) item = atomicAdd(&hdr->next_item, 1);
            item = __shfl_sync(0xffffffffu, item, 0);
            if (item >= n_items) break;
            const int rank = item / (NVT * d.H), hh = (item / NVT) % d.H, vtt = item % NVT;
            const int s = order[rank];
            const int c0 = seq_first[s], nch = seq_first[s + 1] - c0;
            if (nch == 0) {  // empty sequence: the state passes through unchanged
                if (hT) {
                    const size_t base = ((size_t)s * d.H + hh) * DK;
                    for (int e = lane; e < DK * NV; e += 32) {
                        const size_t off = (base + e / NV) * DV + vtt * NV + e % NV;
                        hT[off] = h0 ? h0[off] : 0.f;
                    }
                }
                continue;
            }
            for (int j = 0; j < nch; ++j, ++gj) {
                const int st = gj % kStages;
                if (lane == 0) {
                    if (gj >= kStages &&
                        !ptx::mbar_wait_or_abort(&sm.empty[st], ((gj / kStages) - 1) & 1, abort)) {
                        raise_error(ws, abort);
                        okp = false;
                    } else {
                        const int4 chk = chunks[c0 + j];
                        sm.st[st].item = make_int4(s, hh, vtt, j);
                        sm.st[st].info = make_int4(nch, chk.y, chk.z, 0);
                        const uint8_t* fb = ws + W.factors + ((size_t)(c0 + j) * d.H + hh) * W.factor_bytes;
                        ptx::mbar_arrive_expect_tx(&sm.full[st], main_bytes + u_bytes + gl_bytes);
                        ptx::bulk_g2s(sm.st[st].WQ, fb + F.wq, main_bytes, &sm.full[st]);
                        ptx::bulk_g2s(sm.st[st].U0, fb + F.u0 + (size_t)vtt * u_bytes, u_bytes,
                                      &sm.full[st]);
                        ptx::bulk_g2s(sm.st[st].GL, fb + F.gl, gl_bytes, &sm.full[st]);
                    }
                }
                okp = __shfl_sync(0xffffffffu, okp, 0);
                if (!okp) break;
            }
        }
        if (lane == 0) {
            if (okp) {  // end marker: a stage with no copies that tells the others to stop
                const int st = gj % kStages;
                if (gj >= kStages &&
                    !ptx::mbar_wait_or_abort(&sm.empty[st], ((gj / kStages) - 1) & 1, abort)) {
                    raise_error(ws, abort);
                } else {
                    sm.st[st].info = make_int4(0, 0, 0, 1);
                    ptx::mbar_arrive(&sm.full[st]);
                }
            } else {  // let copies already in flight land before the CTA leaves
                volatile int never = 0;
                const int first = gj - kStages < 0 ? 0 : gj - kStages;
                for (int k2 = first; k2 < gj; ++k2)  // stages issued so far
                    ptx::mbar_wait_or_abort(&sm.full[k2 % kStages], (k2 / kStages) & 1, &never);
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ GEMM3 issue
        if (lane == 0) {
            const uint32_t uop = ptx::smem_u32(sm.Uop);
            constexpr uint32_t id_o = ptx::idesc_bf16(128, NV) | kBMajorMN;
            for (int gj = 0;; ++gj) {
                const int st = gj % kStages;
                if (!ptx::mbar_wait_or_abort(&sm.full[st], (gj / kStages) & 1, abort)) break;
                if (sm.st[st].info.w) break;  // end marker
                if (!ptx::mbar_wait_or_abort(&sm.uready, gj & 1, abort)) break;
                ptx::tc_fence_after();
                // rows 64-127 of this A operand are the P tile (k-block stride 1 KB)
                const uint32_t pa = ptx::smem_u32(sm.st[st].P) - 1024;
                const uint32_t d1 = tmem + kColD1 + (uint32_t)(gj & 1) * NV;
                ptx::mma_chain<kChunk / 16>(d1, ptx::smem_desc(pa, 1024, 128), 2048,  // D1 += P U
                                            ptx::smem_desc(uop, (NV / 8) * 128, 128),
                                            2 * (NV / 8) * 128, id_o, true);
                ptx::mma_commit(&sm.d3[gj & 1]);
                ptx::mma_commit(&sm.empty[st]);
            }
            volatile int never = 0;  // its MMAs complete before TMEM is released
            ptx::mma_commit(&sm.fin3);
            ptx::mbar_wait_or_abort(&sm.fin3, 0, &never);
        }
    } else {
        // ------------------------------------------------ epilogue + MMA issue
        const int w = warp, l = lane;
        const uint32_t lane_base = (uint32_t)(32 * w) << 16;
        const int ch = acc_row<DK>(w, l);     // key channel of this thread's state row
        const int ur = 32 * w + l;            // D1 row (lane): w S rows 0-63, output rows 64-127
        const uint32_t sop = ptx::smem_u32(sm.Sop), uop32 = ptx::smem_u32(sm.Uop32);
        constexpr uint32_t id_w = ptx::idesc_bf16(128, NV) | kAMajorMN | kBMajorMN;
        constexpr uint32_t id_k = ptx::idesc_tf32(DK, NV);   // both K-major
        float S[NV];
#pragma unroll
        for (int n = 0; n < NV; ++n) S[n] = 0.f;
        // Exits are collective: a failed wait in any epilogue thread is folded into
        // the next named-barrier reduction, so all 128 threads leave the loop at the
        // same point and none is left waiting at a barrier.
        bool ok = true;
        bool have_prev = false;
        int4 prev_row = make_int4(0, 0, 0, 0);   // {first token row, rows, head, value tile}
        for (int gj = 0; ok; ++gj) {
            const int st = gj % kStages;
            bool okl = __all_sync(0xffffffffu,
                                  ptx::mbar_wait_or_abort(&sm.full[st], (gj / kStages) & 1, abort));
            ok = epi_sync_and(okl);
            if (!ok) break;
            const int4 it = sm.st[st].item, info = sm.st[st].info;
            const bool end = info.w != 0;
            // -------- a new item: its initial state into S and the bf16 copy
            if (!end && it.w == 0) {
                if (ch >= 0) {
                    const size_t srow = ((size_t)it.x * d.H + it.y) * DK + ch;
#pragma unroll
                    for (int n = 0; n < NV; n += 4) {
                        float4 v4 = h0 ? *reinterpret_cast<const float4*>(&h0[srow * DV + it.z * NV + n])
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                        S[n] = v4.x; S[n + 1] = v4.y; S[n + 2] = v4.z; S[n + 3] = v4.w;
                    }
#pragma unroll
                    for (int nb = 0; nb < NV; nb += 8)
                        *reinterpret_cast<uint4*>(&sm.Sop[nmaj_index<NV>(nb, ch)]) =
                            make_uint4(pack_bf16(S[nb], S[nb + 1]), pack_bf16(S[nb + 2], S[nb + 3]),
                                       pack_bf16(S[nb + 4], S[nb + 5]), pack_bf16(S[nb + 6], S[nb + 7]));
                }
                ptx::fence_proxy_async_smem();
                epi_sync_and(true);
            }
            // -------- issue GEMM1 of this step: D1[gj & 1] = [w ; QG] S
            if (!end && tid == 0) {
                ptx::tc_fence_after();
                const uint32_t wa = ptx::smem_u32(sm.st[st].WQ);
                ptx::mma_chain<DK / 16>(tmem + kColD1 + (uint32_t)(gj & 1) * NV,
                                        ptx::smem_desc(wa, 128, (DK / 8) * 128), 256,
                                        ptx::smem_desc(sop, (NV / 8) * 128, 128),
                                        2 * (NV / 8) * 128, id_w, false);
                ptx::mma_commit(&sm.d1);
            }
            if (w >= 2) {
                // -------- warps 2-3: output of the previous step (overlaps GEMM1)
                if (have_prev) {
                    okl = __all_sync(0xffffffffu, ptx::mbar_wait_or_abort(
                                                      &sm.d3[(gj - 1) & 1], ((gj - 1) >> 1) & 1, abort));
                    if (okl) {
                        ptx::tc_fence_after();
                        float acc[NV];
                        tmem_ldnv<NV>(tmem + lane_base + kColD1 + (uint32_t)((gj - 1) & 1) * NV, acc);
                        const int orow = ur - kChunk;
                        if (orow < prev_row.y)
                            store_row<NV>(o + ((size_t)(prev_row.x + orow) * d.H + prev_row.z) * DV +
                                          prev_row.w * NV,
                                      acc, scale);
                    }
                }
            } else if (!end) {
                // -------- warps 0-1: U = u - (w S)  ->  Uop
                // (Uop is overwritten only once the previous step's GEMM3 has read it)
                bool okw = !have_prev || ptx::mbar_wait_or_abort(&sm.d3[(gj - 1) & 1],
                                                                 ((gj - 1) >> 1) & 1, abort);
                okw = okw && ptx::mbar_wait_or_abort(&sm.d1, gj & 1, abort);
                okl = __all_sync(0xffffffffu, okw);
                if (okl) {
                    ptx::tc_fence_after();
                    float acc[NV];
                    tmem_ldnv<NV>(tmem + lane_base + kColD1 + (uint32_t)(gj & 1) * NV, acc);
                    const float4* u0 = reinterpret_cast<const float4*>(sm.st[st].U0);
                    float U[NV];
#pragma unroll
                    for (int n4 = 0; n4 < NV / 4; ++n4) {
                        const float4 a = u0[n4 * kChunk + ur];
                        U[4 * n4] = a.x - acc[4 * n4];
                        U[4 * n4 + 1] = a.y - acc[4 * n4 + 1];
                        U[4 * n4 + 2] = a.z - acc[4 * n4 + 2];
                        U[4 * n4 + 3] = a.w - acc[4 * n4 + 3];
                    }
#pragma unroll
                    for (int nb = 0; nb < NV; nb += 8)
                        *reinterpret_cast<uint4*>(&sm.Uop[nmaj_index<NV>(nb, ur)]) = make_uint4(
                            pack_bf16(U[nb], U[nb + 1]), pack_bf16(U[nb + 2], U[nb + 3]),
                            pack_bf16(U[nb + 4], U[nb + 5]), pack_bf16(U[nb + 6], U[nb + 7]));
#pragma unroll
                    for (int n = 0; n < NV; ++n) sm.Uop32[u32_index(n, ur)] = U[n];
                }
            }
            if (end) {
                ok = epi_sync_and(okl);
                break;
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ok = epi_sync_and(okl);
            if (!ok) break;
            // -------- issue GEMM2 (serial path); warp 5 issues GEMM3 (output)
            if (tid == 0) {
                ptx::tc_fence_after();
                ptx::mbar_arrive(&sm.uready);
                const uint32_t ka = ptx::smem_u32(sm.st[st].KT);
                const uint64_t a0 = ptx::smem_desc(ka, (DK / 8) * 128, 128);
                const uint64_t b0 = ptx::smem_desc(uop32, kU32Lbo, kU32Sbo);
#pragma unroll
                for (int kk = 0; kk < kChunk / 8; ++kk)  // D2 = KT U, tf32, K = 8 per step
                    ptx::mma_tf32(tmem + kColD2, a0 + (uint64_t)((kk * 2 * (DK / 8) * 128) >> 4),
                                  b0 + (uint64_t)((kk * 2 * kU32Lbo) >> 4), id_k, kk > 0);
                ptx::mma_commit(&sm.d2);
                ptx::mma_commit(&sm.empty[st]);
            }
            // -------- S <- GL * S + D2  ->  Sop (GEMM1 of this step, its one
            //          reader, completed before the barrier above)
            okl = __all_sync(0xffffffffu, ptx::mbar_wait_or_abort(&sm.d2, gj & 1, abort));
            if (okl) {
                ptx::tc_fence_after();
                float acc[NV];
                tmem_ldnv<NV>(tmem + lane_base + kColD2, acc);
                if (ch >= 0) {
                    const float gl = sm.st[st].GL[ch];
                    __nv_bfloat16* so = sm.Sop;
#pragma unroll
                    for (int nb = 0; nb < NV; nb += 8) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) S[nb + e] = fmaf(gl, S[nb + e], acc[nb + e]);
                        *reinterpret_cast<uint4*>(&so[nmaj_index<NV>(nb, ch)]) =
                            make_uint4(pack_bf16(S[nb], S[nb + 1]), pack_bf16(S[nb + 2], S[nb + 3]),
                                       pack_bf16(S[nb + 4], S[nb + 5]), pack_bf16(S[nb + 6], S[nb + 7]));
                    }
                    if (hT && it.w == info.x - 1) {  // the item's last chunk: its final state
                        const size_t srow = ((size_t)it.x * d.H + it.y) * DK + ch;
#pragma unroll
                        for (int n = 0; n < NV; n += 4)
                            *reinterpret_cast<float4*>(&hT[srow * DV + it.z * NV + n]) =
                                make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ok = epi_sync_and(okl);
            if (ok && tid == 0) ptx::mbar_arrive(&sm.empty[st]);  // U0, GL of this stage read
            prev_row = make_int4(info.y, info.z, it.y, it.z);
            have_prev = true;
        }
        if (!ok) raise_error(ws, abort);
        if (tid == 0) {  // every issued MMA completes before TMEM is released
            volatile int never = 0;
            ptx::mma_commit(&sm.fin);
            ptx::mbar_wait_or_abort(&sm.fin, 0, &never);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int DK, int DV, int NV, typename TOut>
cudaError_t launch_t(const Dims& d, const float* h0, float scale, void* o, float* hT, uint8_t* ws,
                     cudaStream_t stream) {
    auto kern = chain_tc_kernel<DK, DV, NV, TOut>;
    const size_t smem = sizeof(ChainSmem<DK, NV>);
    static_assert(sizeof(ChainSmem<DK, NV>) <= 227 * 1024, "state kernel shared memory");
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const long long items = (long long)d.N * d.H * (DV / NV);
    if (items == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(items < num_sms() ? items : num_sms());  // persistent
    kern<<<grid, kThreads, smem, stream>>>(d, h0, scale, static_cast<TOut*>(o), hT, ws);
    return cudaGetLastError();
}

// 64-column value tiles once 32-column chains outnumber the SMs (half the chains,
// twice the work per MMA issue); 16-column tiles while twice the 32-column chains
// still fit on the SMs (each chain is latency-bound, so more of them run at once);
// 32-column tiles in between.
template <int DK, int DV, typename TOut>
cudaError_t launch_nv(const Dims& d, const float* h0, float scale, void* o, float* hT, uint8_t* ws,
                      cudaStream_t stream) {
    const int nv = split_nv_for(d);
    if (nv == 64) return launch_t<DK, DV, 64, TOut>(d, h0, scale, o, hT, ws, stream);
    if (nv == 16) return launch_t<DK, DV, 16, TOut>(d, h0, scale, o, hT, ws, stream);
    return launch_t<DK, DV, 32, TOut>(d, h0, scale, o, hT, ws, stream);
}

}  // namespace

int split_nv_for(const Dims& d) {
    const long long chains32 = (long long)d.N * d.H * (d.dv / 32);
    if (chains32 > num_sms()) return 64;
    if (2 * chains32 <= num_sms()) return 16;
    return 32;
}

cudaError_t launch_chain(const Dims& d, bool qkv_bf16, const float* h0, float scale, void* o,
                         float* hT, uint8_t* ws, cudaStream_t stream) {
#define KDA_CHAIN_CASE(DK_, DV_)                                                              \
    if (d.dk == DK_ && d.dv == DV_)                                                           \
        return qkv_bf16 ? launch_nv<DK_, DV_, __nv_bfloat16>(d, h0, scale, o, hT, ws, stream) \
                        : launch_nv<DK_, DV_, float>(d, h0, scale, o, hT, ws, stream);
    KDA_CHAIN_CASE(64, 64)
    KDA_CHAIN_CASE(64, 128)
    KDA_CHAIN_CASE(128, 64)
    KDA_CHAIN_CASE(128, 128)
#undef KDA_CHAIN_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
