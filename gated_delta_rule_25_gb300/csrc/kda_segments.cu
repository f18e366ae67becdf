// The scan of the segmented chains (split pipeline, few long chains): between the
// two segment passes, every middle segment's map F_k and state from zero Z_k (both
// written by pass A) give the segments' start states, E_{k+1} = F_k E_k + Z_k.
#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

namespace {

constexpr int kCDK = 128, kCDV = 128;  // the head dimensions segments apply to

// The scan between the passes: for every chain with three or more segments, the
// start state of segment k + 1 is F_k E_k + Z_k (k = 1 .. segments - 2), E_1 being
// the first segment's final state; Z_k is overwritten by the result.  The value
// columns are independent, so each CTA takes one 16-column tile of one chain and
// walks its segments in order.  F_k^T arrives in shared memory by one bulk copy (two
// buffers: the maps do not depend on the scan, so the next one loads while a step
// computes; its rows are padded to dk + 8 floats when the map task writes it, so
// that the copy lands conflict-free for the fragment loads) and the tile stays in
// shared memory (rows padded to 24 floats) already split into its tf32 high part and
// remainder, written once per step instead of converted by every warp.  Each step is
// F_k E_k on the tensor cores (mma.sync m16n8k8 on tf32 operands, each split into a
// tf32 high part and the rounding remainder, three products per k-step: about fp32
// accuracy), warp w taking rows 16 w .. 16 w + 15 and both 8-column halves of the
// tile; Z_k, loaded a step ahead, is added in fp32.
constexpr int kScanCols = 16, kScanThreads = 256, kFBufs = 2;
constexpr int kFLd = kCDK + kMapPad;     // padded row of F^T (136: bank offset 8 per row)
constexpr int kPLd = kScanCols + 8;      // padded row of the tile (24: bank offset 24 per row)
struct __align__(16) ScanSmem {
    float FT[kFBufs][kCDK * kFLd];
    uint32_t phi[kCDK * kPLd], plo[kCDK * kPLd];  // the tile: tf32 high part, remainder
    uint64_t full[kFBufs];
    int abort;
};

__device__ __forceinline__ uint32_t tf32_bits(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// x = hi + lo with hi = x rounded to tf32 and lo the remainder rounded to tf32.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_bits(x);
    lo = tf32_bits(x - __uint_as_float(hi));
}
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kScanThreads) seg_scan_kernel(Dims d, uint8_t* __restrict__ ws) {
    constexpr int DK = kCDK, DV = kCDV, kTiles = DV / kScanCols;
    constexpr uint32_t FB = DK * kFLd * 4;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(smem_raw);
    const WsLayout W(d);
    Header* hdr = reinterpret_cast<Header*>(ws + W.header);
    if (!hdr->seg) return;
    const int i = (int)blockIdx.x / kTiles, col0 = kScanCols * ((int)blockIdx.x % kTiles);
    if (i >= hdr->seg_ns) return;
    const int4 e = reinterpret_cast<const int4*>(ws + W.seg_scan)[i];  // {pair, E slot, F slot, segments}
    const int steps = e.w - 2;
    float* E = reinterpret_cast<float*>(ws + W.seg_e);
    const float* FT = reinterpret_cast<const float*>(ws + W.seg_f);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3, r0 = 16 * warp;  // fragment row group, k index; the warp's rows
    uint32_t issued[kFBufs] = {};
    if (tid == 0) {
        for (int bb = 0; bb < kFBufs; ++bb) ptx::mbar_init(&sm.full[bb], 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
        // The maps and Z of the later steps into L2 now (pass A's factor reads may have
        // pushed them out), each by one of the chain's tile CTAs.
        const int tile = (int)blockIdx.x % kTiles;
        for (int k = kFBufs + 1 + tile; k <= steps; k += kTiles) {
            ptx::bulk_prefetch_l2(FT + (size_t)(e.z + k - 1) * DK * kFLd, FB);
            ptx::bulk_prefetch_l2(E + (size_t)(e.y + k) * DK * DV, DK * DV * 4);
        }
        for (int k = 1; k <= kFBufs && k <= steps; ++k) {
            ptx::mbar_arrive_expect_tx(&sm.full[k - 1], FB);
            ptx::bulk_g2s(sm.FT[k - 1], FT + (size_t)(e.z + k - 1) * DK * kFLd, FB, &sm.full[k - 1]);
            ++issued[k - 1];
        }
    }
    for (int x = tid; x < DK * kScanCols; x += kScanThreads) {
        const int at = (x / kScanCols) * kPLd + x % kScanCols;
        split_tf32(E[(size_t)e.y * DK * DV + (size_t)(x / kScanCols) * DV + col0 + x % kScanCols], sm.phi[at],
                   sm.plo[at]);
    }
    __syncthreads();
    bool ok = true;
    // this lane's outputs: rows r0 + gq (+ 8), columns 8 nt + 2 tq (+ 1); Z of the next
    // step is loaded while a step computes
    float2 zn[2][2];
    auto load_z = [&](int k) {
        const float* Ek = E + (size_t)(e.y + k) * DK * DV + col0;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                zn[nt][h] = *reinterpret_cast<const float2*>(Ek + (size_t)(r0 + gq + 8 * h) * DV + 8 * nt + 2 * tq);
    };
    if (steps >= 1) load_z(1);
    for (int k = 1; k <= steps; ++k) {
        const int b = (k - 1) % kFBufs;
        float* Ek = E + (size_t)(e.y + k) * DK * DV + col0;
        float2 z[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) z[nt][h] = zn[nt][h];
        if (k < steps) load_z(k + 1);
        ok = __syncthreads_and(ptx::mbar_wait_or_abort(&sm.full[b], ((k - 1) / kFBufs) & 1u, &sm.abort));
        if (!ok) break;
        const float* F = sm.FT[b];
        // three accumulators per column half and k parity (the three products of a
        // k-step; even and odd k-steps), so that the dependent chains of tensor-core
        // operations are a sixth as long
        float acc[2][2][3][4] = {};
#pragma unroll 2
        for (int k2 = 0; k2 < DK / 16; ++k2) {
#pragma unroll
            for (int par = 0; par < 2; ++par) {
                const int m0 = 16 * k2 + 8 * par;
                // A = F (rows r, k = m): F[r][m] = F^T[m][r]
                const float af[4] = {F[(m0 + tq) * kFLd + r0 + gq], F[(m0 + tq) * kFLd + r0 + gq + 8],
                                     F[(m0 + tq + 4) * kFLd + r0 + gq], F[(m0 + tq + 4) * kFLd + r0 + gq + 8]};
                uint32_t ahi[4], alo[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) split_tf32(af[j], ahi[j], alo[j]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    // B = the tile (k = m, n = column), already split
                    const int at0 = (m0 + tq) * kPLd + 8 * nt + gq, at1 = at0 + 4 * kPLd;
                    const uint32_t b0h = sm.phi[at0], b0l = sm.plo[at0], b1h = sm.phi[at1], b1l = sm.plo[at1];
                    mma_tf32_16x8x8(acc[nt][par][0], alo, b0h, b1h);
                    mma_tf32_16x8x8(acc[nt][par][1], ahi, b0l, b1l);
                    mma_tf32_16x8x8(acc[nt][par][2], ahi, b0h, b1h);
                }
            }
        }
        __syncthreads();  // every warp has read the previous start state and F buffer b
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = r0 + gq + 8 * h, col = 8 * nt + 2 * tq;
                const int i0 = 2 * h, i1 = 2 * h + 1;
                auto sum = [&](int i) {
                    return (acc[nt][0][2][i] + acc[nt][1][2][i]) +
                           ((acc[nt][0][0][i] + acc[nt][0][1][i]) + (acc[nt][1][0][i] + acc[nt][1][1][i]));
                };
                const float2 v = make_float2(sum(i0) + z[nt][h].x, sum(i1) + z[nt][h].y);
                split_tf32(v.x, sm.phi[row * kPLd + col], sm.plo[row * kPLd + col]);
                split_tf32(v.y, sm.phi[row * kPLd + col + 1], sm.plo[row * kPLd + col + 1]);
                *reinterpret_cast<float2*>(Ek + (size_t)row * DV + col) = v;
            }
        if (tid == 0 && k + kFBufs <= steps) {  // the map kFBufs steps ahead into the buffer just read
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive_expect_tx(&sm.full[b], FB);
            ptx::bulk_g2s(sm.FT[b], FT + (size_t)(e.z + k + kFBufs - 1) * DK * kFLd, FB, &sm.full[b]);
            ++issued[b];
        }
        __syncthreads();  // the new start state complete
    }
    if (!ok && tid == 0) {  // a copy did not land in time: report, and let those in flight land
        atomicOr(&hdr->error, kDevErrTimeout);
        volatile int never = 0;
        for (int bb = 0; bb < kFBufs; ++bb)
            if (issued[bb]) ptx::mbar_wait_or_abort(&sm.full[bb], (issued[bb] - 1) & 1u, &never);
    }
}

}  // namespace

cudaError_t launch_seg_scan(const Dims& d, uint8_t* ws, cudaStream_t stream) {
    if (!seg_layout_applies(d)) return cudaErrorInvalidValue;
    const long long pairs = (long long)d.N * d.H;
    if (pairs == 0) return cudaSuccess;
    const size_t smem = sizeof(ScanSmem);
    cudaError_t e = ensure_smem(seg_scan_kernel, smem);
    if (e != cudaSuccess) return e;
    seg_scan_kernel<<<(unsigned)(pairs * (kCDV / kScanCols)), kScanThreads, smem, stream>>>(d, ws);
    return cudaGetLastError();
}

}  // namespace kda
