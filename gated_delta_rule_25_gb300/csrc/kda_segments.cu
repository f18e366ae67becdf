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
// walks its segments in order, in fp32: F_k^T arrives in shared memory by one bulk
// copy (two buffers: the maps do not depend on the scan, so the next one loads
// while a step computes) and the tile stays in shared memory.  The sum over m is
// split in four quarters over the CTA's 16 warps (enough warps to hide the shared
// memory latency); in each quarter a thread accumulates a 4 x 4 block (per m, a
// float4 of F^T's row m and one of the tile's row m: conflict-free and broadcast),
// and the four partial blocks are added with Z_k through shared memory.
constexpr int kScanCols = 16, kScanThreads = 512, kScanK = 4;
constexpr int kPrevLd = kScanCols + 4;  // padded rows: the output threads' row-wise writes hit distinct banks
struct __align__(16) ScanSmem {
    float FT[2][kCDK * kCDK];
    float prev[kCDK][kPrevLd];
    // partial 4 x 4 blocks: [quarter][column group][row group][4 float4], the float4 of
    // block row r at position r ^ ((row group / 2) & 3), so that the 8 threads of a
    // quarter warp store to distinct banks
    float part[kScanK][kScanCols / 4][kCDK / 4][16];
    uint64_t full[2];
    int abort;
};

__global__ void __launch_bounds__(kScanThreads) seg_scan_kernel(Dims d, uint8_t* __restrict__ ws) {
    constexpr int DK = kCDK, DV = kCDV, kTiles = DV / kScanCols, kM = DK / kScanK;
    constexpr uint32_t FB = DK * DK * 4;
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
    const int tid = threadIdx.x;
    const int kq = tid >> 7, rg = tid & 31, cg = (tid >> 5) & 3;  // m quarter; rows 4 rg .., columns 4 cg ..
    const int orow = tid & (DK - 1), ocol = 4 * (tid >> 7);          // the output float4 of this thread
    const int swz = (rg >> 1) & 3, oswz = ((orow >> 2) >> 1) & 3;
    uint32_t issued[2] = {0, 0};
    if (tid == 0) {
        ptx::mbar_init(&sm.full[0], 1);
        ptx::mbar_init(&sm.full[1], 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
        // The maps and Z of the later steps into L2 now (pass A's factor reads may have
        // pushed them out), each by one of the chain's tile CTAs.
        const int tile = (int)blockIdx.x % kTiles;
        for (int k = 3 + tile; k <= steps; k += kTiles) {
            ptx::bulk_prefetch_l2(FT + (size_t)(e.z + k - 1) * DK * DK, FB);
            ptx::bulk_prefetch_l2(E + (size_t)(e.y + k) * DK * DV, FB);
        }
        for (int k = 1; k <= 2 && k <= steps; ++k) {
            ptx::mbar_arrive_expect_tx(&sm.full[k - 1], FB);
            ptx::bulk_g2s(sm.FT[k - 1], FT + (size_t)(e.z + k - 1) * DK * DK, FB, &sm.full[k - 1]);
            ++issued[k - 1];
        }
    }
    *reinterpret_cast<float4*>(&sm.prev[orow][ocol]) =
        *reinterpret_cast<const float4*>(E + (size_t)e.y * DK * DV + (size_t)orow * DV + col0 + ocol);
    __syncthreads();
    bool ok = true;
    for (int k = 1; k <= steps; ++k) {
        const int b = (k - 1) & 1;
        float* Ek = E + (size_t)(e.y + k) * DK * DV + (size_t)orow * DV + col0 + ocol;
        const float4 z = *reinterpret_cast<const float4*>(Ek);
        ok = __syncthreads_and(ptx::mbar_wait_or_abort(&sm.full[b], ((k - 1) >> 1) & 1u, &sm.abort));
        if (!ok) break;
        float acc[4][4] = {};
        const float* ft = sm.FT[b] + kq * kM * DK + 4 * rg;
        const float* pv = &sm.prev[kq * kM][4 * cg];
        // the loads of m + 1 are in flight while m's 16 products run
        float4 f = *reinterpret_cast<const float4*>(ft), p = *reinterpret_cast<const float4*>(pv);
#pragma unroll 4
        for (int m = 0; m < kM; ++m) {
            const float fr[4] = {f.x, f.y, f.z, f.w}, pc[4] = {p.x, p.y, p.z, p.w};
            if (m + 1 < kM) {
                f = *reinterpret_cast<const float4*>(ft + (m + 1) * DK);
                p = *reinterpret_cast<const float4*>(pv + (m + 1) * kPrevLd);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(fr[r], pc[c], acc[r][c]);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(&sm.part[kq][cg][rg][4 * (r ^ swz)]) =
                make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        __syncthreads();  // every partial block written; the previous start state and F buffer b read
        float4 v = z;
#pragma unroll
        for (int q = 0; q < kScanK; ++q) {
            const float4 pp = *reinterpret_cast<const float4*>(
                &sm.part[q][ocol >> 2][orow >> 2][4 * ((orow & 3) ^ oswz)]);
            v.x += pp.x; v.y += pp.y; v.z += pp.z; v.w += pp.w;
        }
        *reinterpret_cast<float4*>(&sm.prev[orow][ocol]) = v;
        *reinterpret_cast<float4*>(Ek) = v;
        if (tid == 0 && k + 2 <= steps) {  // the map after next into the buffer just read
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive_expect_tx(&sm.full[b], FB);
            ptx::bulk_g2s(sm.FT[b], FT + (size_t)(e.z + k + 1) * DK * DK, FB, &sm.full[b]);
            ++issued[b];
        }
        __syncthreads();  // the new start state complete; the partial blocks read
    }
    if (!ok && tid == 0) {  // a copy did not land in time: report, and let those in flight land
        atomicOr(&hdr->error, kDevErrTimeout);
        volatile int never = 0;
        for (int b = 0; b < 2; ++b)
            if (issued[b]) ptx::mbar_wait_or_abort(&sm.full[b], (issued[b] - 1) & 1u, &never);
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
