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
constexpr int kMaxGrid = 1024;  // fused grids of up to this many CTAs

// Per-step times of the state kernels, measured on GB300 (us): a 128-column chain
// step (the segment passes' tasks too), and a 64 / 32 / 16-column tile step.
constexpr float kStep128 = 2.5f;
__host__ __device__ inline float tile_step(int nv) { return nv == 64 ? 2.0f : (nv == 32 ? 1.55f : 1.42f); }
// Predicted time of the tiled state kernel: its items are taken longest first, so
// it is bound by the longest chain or by its share of all the steps.
__host__ __device__ inline float tiled_time(int longest, long long steps, int H, int dv, int nv, int sms) {
    const float share = (float)steps * H * (float)(dv / nv) / (float)sms;
    return tile_step(nv) * ((float)longest > share ? (float)longest : share);
}

// Segments of L chunks: a chain of n chunks has ceil(n / L) segments.  Pass A holds
// per (sequence, head) the first segment and two map tasks per middle segment (or
// the whole chain when it has one segment), pass C the segments after the first.
// Both passes must fit one round of CTAs, and the start states the slots.  Time
// (measured on GB300): 2.5 us per step of the longest task of each pass plus about
// 10 us per pass (a task's start and end: tensor memory, barriers, its first
// copies, its final state), and for the scan about 5 us plus 2.6 us per serial step.
struct SegCount {
    int tasks_a, slots, nseg_max, tail_max;
    __host__ __device__ void add(int n, int L, int H) {  // one sequence of n > 0 chunks
        const int ns = (n + L - 1) / L;
        tasks_a += H * (ns >= 2 ? 2 * ns - 3 : 1);
        slots += H * (ns - 1);
        if (ns > nseg_max) nseg_max = ns;
        const int tail = ns >= 3 ? L : (ns == 2 ? n - L : 0);
        if (tail > tail_max) tail_max = tail;
    }
    // predicted time (us), or a negative value where L does not apply
    __host__ __device__ float time(int L, int longest, int empty_tasks, int sms, int slot_cap) const {
        const int cap = sms < kSegTasks - empty_tasks ? sms : kSegTasks - empty_tasks;
        if (nseg_max < 3 || tasks_a > cap || slots > slot_cap) return -1.f;
        const int head = L < longest ? L : longest;
        return kStep128 * (float)(head + tail_max) + 2.f * 10.f + 5.f + 2.6f * (float)(nseg_max - 2);
    }
};

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

// fused_grid > 0: also Header::n_chain, the production order and cleared ready
// flags for a fused kernel of fused_grid CTAs (needs d.N <= kRankMax).  ratio: the
// time to produce one item's factors over the time of one chain step.
// Header::chain128 (split pipeline): c128_mode 0 or 1 sets it as given; 2 (varlen,
// dk = dv = 128) decides between the state kernel with split_nv-column tiles and the
// 128-column chain kernel from their predicted times on these chain lengths.
// seg_len (split pipeline, seg_layout_applies): > 0, segments of that many chunks;
// 0, none; -1, segments where predicted faster than the tiled state kernel (the
// length then chosen here), with the task lists and the scan's list.
__global__ void __launch_bounds__(kThreads) schedule_kernel(Dims d, const int32_t* cu,
                                                            uint8_t* ws, int fused_grid,
                                                            float ratio, int split_nv, int c128_mode,
                                                            int seg_len, int sms) {
    WsLayout L(d);
    Header* hdr = reinterpret_cast<Header*>(ws + L.header);
    int32_t* seq_first = reinterpret_cast<int32_t*>(ws + L.seq_first);
    int4* chunks = reinterpret_cast<int4*>(ws + L.chunks);
    __shared__ int bad;
    __shared__ int warp_sums[kThreads / 32];
    __shared__ int carry;
    // Up to kRankMax sequences the tables are built in shared memory (and copied
    // out), so that no step reads back global memory this kernel has just written.
    __shared__ int s_first[kRankMax + 1], s_order[kRankMax], s_rf[kRankMax + 1];
    const bool small = d.N <= kRankMax;
    int* const sf = small ? s_first : seq_first;  // first chunk of each sequence
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
            hdr->chain128 = 0;
            hdr->seg = 0;
            hdr->seg_na = hdr->seg_nc = hdr->seg_ns = hdr->seg_len = 0;
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
            sf[s] = excl;
            if (small) seq_first[s] = excl;
        }
        __syncthreads();
        if (tid == 0) carry += warp_sums[kThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) {
        sf[d.N] = carry;
        if (small) seq_first[d.N] = carry;
        hdr->error = 0;
        hdr->total_chunks = carry;
        hdr->next_item = 0;
        hdr->n_chain = 0;
        hdr->chain128 = c128_mode == 1 ? 1 : 0;
        hdr->seg = 0;
        hdr->seg_na = hdr->seg_nc = hdr->seg_ns = hdr->seg_len = 0;
    }
    __syncthreads();
    // the chunk table, one thread per chunk: its sequence is the last one whose first
    // chunk is <= c
    for (int c = tid; c < carry; c += kThreads) {
        int lo = 0, hi = d.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sf[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        long long r0;
        int len;
        seq_span(d, cu, lo, r0, len);
        const int j = c - sf[lo];
        const int rows = len - j * kChunk;
        chunks[c] = make_int4(lo, (int)(r0 + (long long)j * kChunk), rows < kChunk ? rows : kChunk, j);
    }
    // Longest chains first: the state kernel maps its CTAs through this order so
    // that a dominant sequence starts at once instead of after the short ones.
    // Stable rank by chunk count for up to kRankMax sequences, identity beyond.
    int32_t* order = reinterpret_cast<int32_t*>(ws + L.order);
    __syncthreads();
    if (small) {
        for (int s = tid; s < d.N; s += kThreads) {
            const int ns = sf[s + 1] - sf[s];
            int rank = 0;
            for (int t = 0; t < d.N; ++t) {
                const int nt = sf[t + 1] - sf[t];
                rank += (nt > ns) || (nt == ns && t < s);
            }
            order[rank] = s;
            s_order[rank] = s;
        }
    } else {
        for (int s = tid; s < d.N; s += kThreads) order[s] = s;
    }
    if ((fused_grid <= 0 && c128_mode != 2 && seg_len == 0) || !small) return;

    // ---- fused pipeline.  Chain r = rank * H + head (one chain per sequence and
    // head); chain CTA x takes chains x, x + n_chain, ... (round k = r / n_chain), so
    // CTA 0 runs the longest chain of every round.  rf: chunks before each rank.
    __syncthreads();  // s_order complete
    __shared__ int s_rc0[kRankMax], s_rcnt[kRankMax];  // first chunk and chunks of each rank
    for (int rk = tid; rk < d.N; rk += kThreads) {
        const int sq = s_order[rk];
        s_rc0[rk] = s_first[sq];
        s_rcnt[rk] = s_first[sq + 1] - s_first[sq];
    }
    __syncthreads();
    auto rc0 = [&](int rk) { return s_rc0[rk]; };
    auto rcntf = [&](int rk) { return s_rcnt[rk]; };
    if (fused_grid <= 0) {
        // ---- split pipeline: which state kernel.  Per-step times measured on GB300:
        // 2.5 us for a 128-column chain step, 2.0 / 1.55 / 1.42 us for a 64 / 32 / 16
        // column one.  The 128-column kernel gives CTA x chains x, x + G, ... (G CTAs;
        // CTA 0, with the longest of each round, finishes last); the tiled kernel takes
        // its (chain, tile) items longest first from a counter, bounded by the longest
        // chain or by its share of all the steps.
        const int H = d.H, R = d.N * d.H;
        const int longest = d.N > 0 ? rcntf(0) : 0;
        const float tnv = tiled_time(longest, carry, H, d.dv, split_nv, sms);
        if (c128_mode == 2) {
            __shared__ int steps128;
            const int G = R < sms ? R : sms;
            if (tid == 0) steps128 = 0;
            __syncthreads();
            if (tid < 32 && G > 0) {
                int sum = 0;
                for (int k = tid; k * G < R; k += 32) sum += rcntf((k * G) / H);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (tid == 0) steps128 = sum;
            }
            __syncthreads();
            if (tid == 0) hdr->chain128 = kStep128 * (float)steps128 < 0.9f * tnv ? 1 : 0;
        }
        if (seg_len == 0 || !seg_layout_applies(d) || L.seg_slots == 0) return;
        // ---- segments (few chains, at most kSegPairs): the length, then the lists
        __shared__ unsigned long long seg_best;
        __shared__ int s_empty;
        if (tid == 0) {
            seg_best = ~0ull;
            int empty = 0;
            for (int rk = 0; rk < d.N; ++rk) empty += rcntf(rk) == 0;
            s_empty = empty * H;
        }
        __syncthreads();
        int Lp = seg_len;
        if (seg_len < 0) {
            for (int Lc = tid + 1; Lc < longest; Lc += kThreads) {
                SegCount sc{0, 0, 0, 0};
                for (int rk = 0; rk < d.N; ++rk)
                    if (rcntf(rk) > 0) sc.add(rcntf(rk), Lc, H);
                const float t = sc.time(Lc, longest, s_empty, sms, L.seg_slots);
                if (t >= 0.f)
                    atomicMin(&seg_best, ((unsigned long long)__float_as_uint(t) << 32) | (unsigned long long)Lc);
            }
            __syncthreads();
            Lp = 0;
            if (seg_best != ~0ull && __uint_as_float((unsigned)(seg_best >> 32)) < 0.85f * tnv)
                Lp = (int)(seg_best & 0xffffffffull);
        }
        if (Lp <= 0) return;
        // The lists, one thread per (rank, head) pair in rank order: its task counts,
        // their exclusive prefixes (thread 0, at most kSegPairs pairs), then its tasks.
        __shared__ int s_pa[kSegPairs + 1], s_pc[kSegPairs + 1], s_pe[kSegPairs + 1], s_pf[kSegPairs + 1],
            s_ps[kSegPairs + 1], s_pz[kSegPairs + 1];
        __shared__ int s_plan_ok;
        const int P = d.N * H;
        if (tid == 0) {
            SegCount sc{0, 0, 0, 0};  // a length given by the host was checked there with the same counts
            for (int rk = 0; rk < d.N; ++rk)
                if (rcntf(rk) > 0) sc.add(rcntf(rk), Lp, H);
            s_plan_ok = sc.time(Lp, longest, s_empty, sms, L.seg_slots) >= 0.f;
            if (!s_plan_ok) hdr->error |= kDevErrPlan;
            int a = 0, c = 0, e = 0, f = 0, sn = 0, z = 0;
            for (int p = 0; p < P; ++p) {
                s_pa[p] = a; s_pc[p] = c; s_pe[p] = e; s_pf[p] = f; s_ps[p] = sn; s_pz[p] = z;
                const int n = rcntf(p / H), nseg = (n + Lp - 1) / Lp;
                if (n == 0) {
                    ++z;
                    continue;
                }
                a += nseg >= 2 ? 2 * nseg - 3 : 1;
                c += nseg - 1;
                e += nseg - 1;
                f += nseg >= 2 ? nseg - 2 : 0;
                sn += nseg >= 3;
            }
            s_pa[P] = a; s_pc[P] = c; s_pe[P] = e; s_pf[P] = f; s_ps[P] = sn; s_pz[P] = z;
        }
        __syncthreads();
        if (!s_plan_ok) return;
        int4* ta = reinterpret_cast<int4*>(ws + L.seg_a);
        int4* tc = reinterpret_cast<int4*>(ws + L.seg_c);
        int4* tscan = reinterpret_cast<int4*>(ws + L.seg_scan);
        for (int p = tid; p < P; p += kThreads) {
            const int rk = p / H, h = p - rk * H, sq = s_order[rk], n = rcntf(rk), c0 = rc0(rk);
            const int pair = sq * H + h;
            if (n == 0) {  // empty sequences last: h_T = h0
                ta[s_pa[P] + s_pz[p]] = make_int4(0, 0, pair, kTaskWhole);
                continue;
            }
            const int nseg = (n + Lp - 1) / Lp, eb = s_pe[p], fb = s_pf[p];
            int na = s_pa[p], nct = s_pc[p];
            if (nseg == 1) {
                ta[na] = make_int4(c0, n, pair, kTaskWhole);
                continue;
            }
            ta[na++] = make_int4(c0, Lp, pair, kTaskHead | (eb << 4));
            for (int k = 1; k + 1 < nseg; ++k) {
                ta[na++] = make_int4(c0 + k * Lp, Lp, pair, kTaskMapF | ((fb + k - 1) << 4));
                ta[na++] = make_int4(c0 + k * Lp, Lp, pair, kTaskMapZ | ((eb + k) << 4));
            }
            for (int k = 1; k < nseg; ++k) {
                const int len = n - k * Lp < Lp ? n - k * Lp : Lp;
                tc[nct++] = make_int4(c0 + k * Lp, len, pair, kTaskTail | ((k == nseg - 1) << 3) | ((eb + k - 1) << 4));
            }
            if (nseg >= 3) tscan[s_ps[p]] = make_int4(pair, eb, fb, nseg);
        }
        if (tid != 0) return;
        const int na = s_pa[P] + s_pz[P], nct = s_pc[P], ns = s_ps[P];
        hdr->seg = 1;
        hdr->seg_na = na;
        hdr->seg_nc = nct;
        hdr->seg_ns = ns;
        hdr->seg_len = Lp;
        return;
    }
    int* const rf = s_rf;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < d.N; base += kThreads) {
        const int rk = base + tid;
        const int e = block_scan(rk < d.N ? rcntf(rk) : 0, warp_sums, &carry);
        if (rk < d.N) rf[rk] = e;
    }
    if (tid == 0) rf[d.N] = carry;
    __syncthreads();
    // n_chain c minimises max(chain steps of CTA 0, ratio * items / (grid - c)): the
    // chain CTAs' critical path against the factor CTAs' share of the items.  CTA 0
    // runs chains 0, c, 2c, ...: steps(c) = sum over rounds k of the count of rank
    // (k c) / H, summed by several threads per candidate (ranks tracked without
    // division).
    __shared__ int steps_s[kMaxGrid + 1];
    __shared__ unsigned long long best;
    const int H = d.H, N = d.N;
    const int R = N * H, items = carry * H;
    const int cmax = R < fused_grid - 1 ? R : fused_grid - 1;
    for (int c = tid; c <= cmax; c += kThreads) steps_s[c] = 0;
    if (tid == 0) best = ~0ull;
    __syncthreads();
    {
        const int split = cmax > 0 ? (kThreads / cmax > 0 ? kThreads / cmax : 1) : 1;
        for (int w = tid; w < cmax * split; w += kThreads) {
            const int c = w % cmax + 1, part = w / cmax;
            const int stride = split * c;  // chains between this thread's rounds
            const int dq = stride / H, dr = stride - dq * H;
            int rk = (part * c) / H, rem = part * c - rk * H, sum = 0;
            for (int r = part * c; r < R; r += stride) {
                sum += rcntf(rk);
                rk += dq;
                rem += dr;
                if (rem >= H) {
                    rem -= H;
                    ++rk;
                }
            }
            atomicAdd(&steps_s[c], sum);
        }
    }
    __syncthreads();
    for (int c = tid + 1; c <= cmax; c += kThreads) {
        const float cost = fmaxf((float)steps_s[c], ratio * (float)items / (float)(fused_grid - c));
        atomicMin(&best, ((unsigned long long)__float_as_uint(cost) << 32) | (unsigned long long)c);
    }
    __syncthreads();
    const int nc = best == ~0ull ? cmax : (int)(best & 0xffffffffull);
    if (tid == 0) hdr->n_chain = nc;

    // Production order: the items of round k (its chains' chunks) come before those
    // of round k + 1, and inside a round step j of every chain comes before step
    // j + 1 (chains in the round's order), so that the chain CTAs find their next
    // chunk published early.  Items are taken in chain order (t, the index there),
    // each thread a run of consecutive ones, walking (rank, head, step) forward;
    // each also clears its ready flag.  32-bit arithmetic throughout (items and
    // chains stay far below 2^31); counts do not increase with the rank.
    int32_t* plist = reinterpret_cast<int32_t*>(ws + L.plist);
    uint32_t* ready = reinterpret_cast<uint32_t*>(ws + L.ready);
    auto before = [&](int x) -> int {  // items of the chains before chain x
        if (x >= R) return items;
        const int rk = x / H;
        return H * rf[rk] + (x - rk * H) * rcntf(rk);
    };
    const int per = (items + kThreads - 1) / kThreads;
    int t = tid * per;
    const int t_end = t + per < items ? t + per : items;
    if (t < t_end) {
        // the rank holding item t: the last rank with H * rf[rank] <= t (its count > 0)
        int lo = 0, hi = N;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (H * rf[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        int rank = lo, len = rcntf(rank);
        const int within = t - H * rf[rank];
        int h = within / len, j = within - h * len;
        int r = rank * H + h;
        int a = r - r % nc, b = a + nc < R ? a + nc : R;
        int a_rank = a / H, Ba = before(a), Bb = before(b);
        for (; t < t_end; ++t) {
            // chains of the round longer than j: a prefix, bounded by the first rank
            // (from a's) whose count is <= j
            int l2 = a_rank, h2 = N;
            while (l2 < h2) {
                const int mid = (l2 + h2) >> 1;
                if (rcntf(mid) <= j) h2 = mid;
                else l2 = mid + 1;
            }
            const int x1 = l2 * H;
            int cnt, Bc;
            if (x1 <= a) {
                cnt = 0;
                Bc = Ba;
            } else if (x1 >= b) {
                cnt = b - a;
                Bc = Bb;
            } else {
                cnt = x1 - a;
                Bc = H * rf[l2];
            }
            // rounds before + steps < j of this round's chains + chains before r at step j
            const int pos = Ba + j * cnt + (Bb - Bc) + (r - a);
            const int c = rc0(rank) + j;
            plist[pos] = c * H + h;
            ready[(size_t)c * H + h] = 0u;
            if (++j == len) {  // the next chain
                j = 0;
                ++r;
                if (++h == H) {
                    h = 0;
                    ++rank;
                    len = rank < N ? rcntf(rank) : 0;
                }
                if (r >= b) {  // the next round
                    a = b;
                    b = a + nc < R ? a + nc : R;
                    a_rank = a / H;
                    Ba = Bb;
                    Bb = before(b);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_schedule(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws, int split_nv,
                            int c128_mode, int seg_len, cudaStream_t stream) {
    schedule_kernel<<<1, kThreads, 0, stream>>>(d, cu_seqlens, ws, 0, 0.f, split_nv, c128_mode, seg_len,
                                                num_sms());
    return cudaGetLastError();
}

// The same prediction as the schedule kernel's, for chains of equal length.
int seg_pick_uniform(const Dims& d) {
    const WsLayout W(d);
    if (!seg_layout_applies(d) || W.seg_slots == 0 || d.N > kRankMax) return 0;
    const int n = (int)(((long long)d.T + kChunk - 1) / kChunk);
    if (n == 0 || d.N == 0) return 0;
    const int sms = num_sms();
    const float tnv = tiled_time(n, (long long)n * d.N, d.H, d.dv, split_nv_for(d), sms);
    float best = -1.f;
    int bestL = 0;
    for (int L = 1; L < n; ++L) {
        SegCount sc{0, 0, 0, 0};
        for (int s = 0; s < d.N; ++s) sc.add(n, L, d.H);
        const float t = sc.time(L, n, 0, sms, W.seg_slots);
        if (t >= 0.f && (best < 0.f || t < best)) {
            best = t;
            bestL = L;
        }
    }
    return best >= 0.f && best < 0.85f * tnv ? bestL : 0;
}

// The same prediction as the schedule kernel's, for chains of equal length.
bool chain128_pick_uniform(const Dims& d) {
    const long long nch = ((long long)d.T + kChunk - 1) / kChunk;  // chunks per chain
    const long long R = (long long)d.N * d.H;
    const int sms = num_sms();
    if (R == 0 || nch == 0) return false;
    const long long G = R < sms ? R : sms;
    const float t128 = kStep128 * (float)(((R + G - 1) / G) * nch);
    return t128 < 0.9f * tiled_time((int)nch, nch * d.N, d.H, d.dv, split_nv_for(d), sms);
}

cudaError_t launch_schedule_fused(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws,
                                  int fused_grid, float production_ratio, cudaStream_t stream) {
    schedule_kernel<<<1, kThreads, 0, stream>>>(d, cu_seqlens, ws, fused_grid, production_ratio, 0, 0, 0, 0);
    return cudaGetLastError();
}

}  // namespace kda
