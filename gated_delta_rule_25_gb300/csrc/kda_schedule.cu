// Chunk schedule: reads the sequence boundaries (cu_seqlens, or the fixed-length
// batch shape) on the device and lays out the list of 64-token chunks that the
// factor and state kernels walk; for the fused pipeline also the split of its CTAs
// between factor production and state chains, and the production order.
// Boundaries are always read from cu_seqlens at run time, never assumed ("NVIDIA
// Kernel Design Agents optimize Kimi Delta Attention", section 03 REWARD HACKING,
// shape and layout hard-coding).
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kThreads = 1024;
constexpr int kPlanThreads = 256;

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

// Exclusive prefix of x over the CTA's threads (in thread order), offset by *carry,
// which then advances by the CTA's total.  Every thread of the CTA calls it.
__device__ int block_scan(int x, int* warp_sums, int* carry) {
    const int tid = threadIdx.x;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if ((tid & 31) >= o) incl += y;
    }
    if ((tid & 31) == 31) warp_sums[tid >> 5] = incl;
    __syncthreads();
    if (tid < 32) {
        int w = warp_sums[tid];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (tid >= o) w += y;
        }
        warp_sums[tid] = w;  // inclusive over warps
    }
    __syncthreads();
    const int excl = *carry + incl - x + ((tid >> 5) ? warp_sums[(tid >> 5) - 1] : 0);
    __syncthreads();
    if (tid == 0) *carry += warp_sums[kThreads / 32 - 1];
    __syncthreads();
    return excl;
}

// fused_grid > 0: also rank_first and Header::n_chain for a fused kernel of
// fused_grid CTAs (needs d.N <= kRankMax).  ratio: the time to produce one item's
// factors over the time of one chain step.
__global__ void __launch_bounds__(kThreads) schedule_kernel(Dims d, const int32_t* cu,
                                                            uint8_t* ws, int fused_grid,
                                                            float ratio) {
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
            hdr->n_chain = 0;
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
        hdr->n_chain = 0;
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
    if (fused_grid <= 0 || d.N > kRankMax) return;

    // ---- fused pipeline.  Chain r = rank * H + head (one chain per sequence and
    // head); chain CTA x takes chains x, x + n_chain, ... (round k = r / n_chain), so
    // CTA 0 runs the longest chain of every round.  rank_first: chunks before each
    // rank in longest-first order.
    int32_t* rank_first = reinterpret_cast<int32_t*>(ws + L.rank_first);
    __syncthreads();  // order complete
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < d.N; base += kThreads) {
        const int rk = base + tid;
        const int n = rk < d.N ? seq_first[order[rk] + 1] - seq_first[order[rk]] : 0;
        const int e = block_scan(n, warp_sums, &carry);
        if (rk < d.N) rank_first[rk] = e;
    }
    if (tid == 0) rank_first[d.N] = carry;
    __syncthreads();
    // n_chain c minimises max(chain steps of CTA 0, ratio * items / (grid - c)):
    // the chain CTAs' critical path against the factor CTAs' share of the items.
    __shared__ unsigned long long best;
    if (tid == 0) best = ~0ull;
    __syncthreads();
    const long long R = (long long)d.N * d.H, items = (long long)carry * d.H;
    const long long cmax = R < fused_grid - 1 ? R : fused_grid - 1;
    for (long long c = tid + 1; c <= cmax; c += kThreads) {
        const long long rounds = (R + c - 1) / c;
        if (rounds > 1024) continue;
        long long steps = 0;
        for (long long k = 0; k < rounds; ++k) {
            const int rk = (int)(k * c / d.H);
            steps += rank_first[rk + 1] - rank_first[rk];
        }
        const float cost = fmaxf((float)steps, ratio * (float)items / (float)(fused_grid - c));
        atomicMin(&best, ((unsigned long long)__float_as_uint(cost) << 32) | (unsigned long long)c);
    }
    __syncthreads();
    if (tid == 0) hdr->n_chain = best == ~0ull ? (int)cmax : (int)(best & 0xffffffffull);
}

// Production order of the fused pipeline: the items of round k (its chains' chunks)
// come before those of round k + 1, and inside a round step j of every chain comes
// before step j + 1 (chains in the round's order), so that the chain CTAs find
// their next chunk published early.  One thread per item, taken in chain order;
// also clears the item's ready flag.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Dims d, uint8_t* ws) {
    const WsLayout L(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + L.header);
    const int nc = hdr->n_chain;
    if (nc <= 0 || hdr->error) return;
    const int H = d.H;
    const int32_t* rf = reinterpret_cast<const int32_t*>(ws + L.rank_first);
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + L.seq_first);
    const int32_t* order = reinterpret_cast<const int32_t*>(ws + L.order);
    int32_t* plist = reinterpret_cast<int32_t*>(ws + L.plist);
    uint32_t* ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    const long long items = (long long)hdr->total_chunks * H;
    const long long t = (long long)blockIdx.x * kPlanThreads + threadIdx.x;
    if (t >= items) return;
    // the rank holding item t: the last rank with H * rf[rank] <= t (its length > 0)
    int lo = 0, hi = d.N;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)H * rf[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    const int rank = lo, len = rf[rank + 1] - rf[rank];
    const long long within = t - (long long)H * rf[rank];
    const int h = (int)(within / len), j = (int)(within % len);
    const long long R = (long long)d.N * H, r = (long long)rank * H + h;
    auto len_of = [&](long long x) { const int rk = (int)(x / H); return rf[rk + 1] - rf[rk]; };
    // items of the chains before chain x (chain order)
    auto before = [&](long long x) -> long long {
        if (x >= R) return items;
        const int rk = (int)(x / H);
        return (long long)H * rf[rk] + (x % H) * (long long)(rf[rk + 1] - rf[rk]);
    };
    const long long a = (r / nc) * nc, b = a + nc < R ? a + nc : R;
    // cnt: chains of the round longer than j (a prefix: lengths do not increase)
    long long l2 = a, h2 = b;
    while (l2 < h2) {
        const long long mid = (l2 + h2) >> 1;
        if (len_of(mid) <= j) h2 = mid;
        else l2 = mid + 1;
    }
    const long long cnt = l2 - a;
    // rounds before + steps < j of this round's chains + chains before r at step j
    const long long pos = before(a) + (long long)j * cnt + (before(b) - before(a + cnt)) + (r - a);
    const int c = seq_first[order[rank]] + j;
    plist[pos] = c * H + h;
    ready[(size_t)c * H + h] = 0u;
}

}  // namespace

cudaError_t launch_schedule(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws,
                            cudaStream_t stream) {
    schedule_kernel<<<1, kThreads, 0, stream>>>(d, cu_seqlens, ws, 0, 0.f);
    return cudaGetLastError();
}

cudaError_t launch_schedule_fused(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws,
                                  int fused_grid, float production_ratio, cudaStream_t stream) {
    schedule_kernel<<<1, kThreads, 0, stream>>>(d, cu_seqlens, ws, fused_grid, production_ratio);
    return cudaGetLastError();
}

cudaError_t launch_plan(const Dims& d, uint8_t* ws, cudaStream_t stream) {
    const WsLayout L(d);
    const long long items = L.cmax * d.H;
    if (items == 0) return cudaSuccess;
    const long long blocks = (items + kPlanThreads - 1) / kPlanThreads;
    plan_kernel<<<(unsigned)blocks, kPlanThreads, 0, stream>>>(d, ws);
    return cudaGetLastError();
}

}  // namespace kda
