// Chunk schedule: reads the sequence boundaries (cu_seqlens, or the fixed-length
// batch shape) on the device and lays out the list of 64-token chunks that the
// factor and state kernels walk.  Boundaries are always read from cu_seqlens at
// run time, never assumed ("NVIDIA Kernel Design Agents optimize Kimi Delta
// Attention", section 03 REWARD HACKING, shape and layout hard-coding).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;
constexpr int kRankMax = 2048;

__device__ inline void seq_span(const Dims& d, const int32_t* cu, int s, long long& row0,
                                int& len) {
    if (d.varlen) {
        row0 = cu[s];
        len = cu[s + 1] - cu[s];
    } else {
        row0 = (long long)s * d.T;
        len = d.T;
    }
}

__global__ void __launch_bounds__(kThreads) schedule_kernel(Dims d, const int32_t* cu,
                                                            uint8_t* ws) {
    WsLayout L(d);
    Header* hdr = reinterpret_cast<Header*>(ws + L.header);
    int32_t* seq_first = reinterpret_cast<int32_t*>(ws + L.seq_first);
    int4* chunks = reinterpret_cast<int4*>(ws + L.chunks);
    __shared__ int bad;
    __shared__ int warp_sums[kThreads / 32];
    __shared__ int carry;
    const int tid = threadIdx.x;
    if (tid == 0) {
        bad = 0;
        carry = 0;
    }
    __syncthreads();
    if (d.varlen) {
        if (tid == 0 && (cu[0] != 0 || cu[d.N] != d.T)) atomicOr(&bad, 1);
        for (int s = tid; s < d.N; s += kThreads)
            if (cu[s + 1] < cu[s]) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (bad) {
        for (int s = tid; s <= d.N; s += kThreads) seq_first[s] = 0;
        int32_t* order = reinterpret_cast<int32_t*>(ws + L.order);
        for (int s = tid; s < d.N; s += kThreads) order[s] = s;
        if (tid == 0) {
            hdr->error = kDevErrCuSeqlens;
            hdr->total_chunks = 0;
            hdr->next_item = 0;
        }
        return;
    }
    // exclusive scan of per-sequence chunk counts, kThreads sequences at a time
    for (int base = 0; base < d.N; base += kThreads) {
        int s = base + tid;
        int n = 0;
        if (s < d.N) {
            long long r0;
            int len;
            seq_span(d, cu, s, r0, len);
            n = (len + kChunk - 1) / kChunk;
        }
        int x = n;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if ((tid & 31) >= o) x += y;
        }
        if ((tid & 31) == 31) warp_sums[tid >> 5] = x;
        __syncthreads();
        if (tid < 32) {
            int w = warp_sums[tid];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, w, o);
                if (tid >= o) w += y;
            }
            warp_sums[tid] = w;  // inclusive over warps
        }
        __syncthreads();
        int excl = carry + x - n + ((tid >> 5) ? warp_sums[(tid >> 5) - 1] : 0);
        if (s < d.N) {
            seq_first[s] = excl;
            long long r0;
            int len;
            seq_span(d, cu, s, r0, len);
            for (int j = 0; j < n; ++j) {
                int rows = len - j * kChunk;
                chunks[excl + j] = make_int4(s, (int)(r0 + (long long)j * kChunk),
                                             rows < kChunk ? rows : kChunk, j);
            }
        }
        __syncthreads();
        if (tid == 0) carry += warp_sums[kThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) {
        seq_first[d.N] = carry;
        hdr->error = 0;
        hdr->total_chunks = carry;
        hdr->next_item = 0;
    }
    // Longest chains first: the state kernel maps its CTAs through this order so
    // that a dominant sequence starts at once instead of after the short ones.
    // Stable rank by chunk count for up to kRankMax sequences, identity beyond.
    int32_t* order = reinterpret_cast<int32_t*>(ws + L.order);
    __syncthreads();
    if (d.N <= kRankMax) {
        for (int s = tid; s < d.N; s += kThreads) {
            const int ns = seq_first[s + 1] - seq_first[s];
            int rank = 0;
            for (int t = 0; t < d.N; ++t) {
                const int nt = seq_first[t + 1] - seq_first[t];
                rank += (nt > ns) || (nt == ns && t < s);
            }
            order[rank] = s;
        }
    } else {
        for (int s = tid; s < d.N; s += kThreads) order[s] = s;
    }
}

}  // namespace

cudaError_t launch_schedule(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws,
                            cudaStream_t stream) {
    schedule_kernel<<<1, kThreads, 0, stream>>>(d, cu_seqlens, ws);
    return cudaGetLastError();
}

}  // namespace kda
