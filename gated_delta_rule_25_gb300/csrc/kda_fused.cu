// Fused pipeline: one persistent launch in which some CTAs produce the per-chunk
// factor blocks (the factor body, items in the schedule kernel's production order) and
// the others run the state recurrence, each over whole (sequence, head) chains
// with all dv value columns at once, consuming every block as soon as its producer
// has published it (a per-item ready flag, release/acquire at GPU scope).  A block
// is then read back while it is still in L2, and the recurrence, latency-bound on
// its own, runs beside the factor production instead of after it ("Autoresearch on
// Kimi Delta Attention", section OPTIMIZATION TRACE: large intermediate surfaces
// written and read back are what such a pipeline avoids).  dk = dv = 128.
//
// The launch is cooperative (every CTA resident at once): chain CTAs wait for
// factor CTAs, never the reverse, and every wait is bounded.
//
// A chain step works on transposes, so that the operands made from the state live
// in tensor memory (the A operand of an MMA may be read from there) instead of
// passing through shared memory: lane n of tensor memory is value column n.  For
// chunk j of a chain (fp32 state S^T, dv x dk, in registers: warp w holds lanes
// 32 (w % 4) .. and channels 32 (w / 4) ..), all products with M = dv:
//   (w S)^T  = S^T w^T         GEMM1a/b  N=64, K=dk, its two channel halves into two
//                                        accumulators (bf16, A = S^T in TMEM)
//   (QG S)^T = S^T QG^T        GEMM1c    N=64, K=dk (the output part)
//   U^T = u^T - (w S)^T                  fp32 into TMEM, and bf16 for GEMM3
//   S^T <- S^T Diag(GL) + U^T KT^T       GEMM2  N=dk, K=64 (tf32, A = U^T in TMEM)
//   O^T = scale ((QG S)^T + U^T P^T)     GEMM3  N=64, K=64 (bf16, A = U^T in TMEM)
// [w; QG], u, KT (with GL) and P arrive by bulk copies into shared memory, each
// part as soon as its slot frees; the output of step j is staged in shared memory
// while GEMM2 of step j + 1 runs and leaves by bulk copies during step j + 2.
#include "kda_factor_body.cuh"

namespace kda {

namespace {

constexpr int kCDK = 128, kCDV = 128;  // the fused pipeline's head dimensions

// Tensor-memory columns of a chain CTA (512 allocated; lane = value column n).
constexpr uint32_t kTS = 0;     // S^T in bf16 (GEMM1's A): channel c at column c / 2
constexpr uint32_t kTXa = 64;   // (w S)^T over channels 0-63, then U^T in tf32 (GEMM2's A)
constexpr uint32_t kTXb = 128;  // (w S)^T over channels 64-127
constexpr uint32_t kTO = 192;   // O^T[b] at 192 + 64 b: (QG S)^T + U^T P^T (the output)
constexpr uint32_t kTD2 = 320;  // D2^T = U^T KT^T, column = channel
constexpr uint32_t kTUB = 448;  // U^T in bf16 (GEMM3's A), 32 columns

struct __align__(1024) ChainRoleSmem {
    __nv_bfloat16 WQ[2 * kChunk * kCDK];   // [w; QG], N-major operand (GEMM1 B)
    float KT[kCDK * kChunk];               // K-major tf32 operand (GEMM2 B)
    __nv_bfloat16 P[2][kChunk * kChunk];   // K-major operand (GEMM3 B), alternate steps
    float GL[2][kCDK];                     // exp(Gamma_last), alternate steps
    float U0[kChunk * kCDV];               // u as [64/4][dv][4] (a float4 of 4 rows per column)
    float otile[kChunk * kCDV];            // one step's output rows (bf16 or fp32), staged
    uint64_t wq_full, kt_full, u_full, p_full[2], d1, d2, d3[2], fin;
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ void chain_raise(uint8_t* ws, volatile int* abort) {
    *abort = 1;
    atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
}

__device__ __forceinline__ void store_out(__nv_bfloat16* p, float x) { *p = __float2bfloat16(x); }
__device__ __forceinline__ void store_out(float* p, float x) { *p = x; }

// A position in this CTA's chains: chain r = rank * H + head (ranks longest first),
// or task r of a segment pass; the CTA takes chains first, first + nc, ...; j is the
// step (chunk) in the chain.
struct ChainPos {
    int r, s, h, c0, len, j;
    int tok0, ntok;  // the chain's first token row and its tokens
    int w;           // segment task: kind | last << 3 | slot << 4 (kTaskWhole otherwise)
};

// A segment pass: its tasks and the segment buffers (dk x dv fp32 each).
struct SegRun {
    const int4* tasks;
    int ntasks;
    float* E;  // segment start states, row-major (and, before the scan, the middle segments' Z)
    float* F;  // the middle segments' maps, transposed: F^T[m][r] = F[r][m], rows of dk + kMapPad
};

// Where a task's chain starts and where its final state goes.
__device__ __forceinline__ bool task_outputs(int w) { return (w & 7) != kTaskMapF && (w & 7) != kTaskMapZ; }

// nc: the chain CTAs (this one is blockIdx.x among them).  use_flags: the factor
// blocks are published as the pipeline runs (fused kernel); false when they were all
// written before this kernel started (the split pipeline's 128-column chain kernel).
// kSeg: the chains are the tasks of a segment pass (seg).
template <typename TOut, bool kSeg = false>
__device__ __forceinline__ void chain_role(const Dims& d, const float* __restrict__ h0, float scale,
                                           TOut* __restrict__ o, float* __restrict__ hT,
                                           uint8_t* __restrict__ ws, uint8_t* smem_raw, int nc,
                                           bool use_flags, const SegRun* seg = nullptr) {
    constexpr int DK = kCDK, DV = kCDV;
    ChainRoleSmem& sm = *reinterpret_cast<ChainRoleSmem*>(smem_raw);
    constexpr uint32_t WQB = 2 * kChunk * DK * 2, KTB = DK * kChunk * 4, PB = kChunk * kChunk * 2,
                       GLB = DK * 4, UB = kChunk * DV * 4;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, g = warp >> 2;
    const int n = 32 * q + lane;  // value column = tensor-memory lane of this thread
    const uint32_t lb = (uint32_t)(32 * q) << 16;
    const WsLayout W(d);
    const FactorLayout F(DK, DV);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    const volatile uint32_t* err = &hdr->error;
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int32_t* order = reinterpret_cast<const int32_t*>(ws + W.order);
    const int4* chunk_tab = reinterpret_cast<const int4*>(ws + W.chunks);
    const uint32_t* ready = reinterpret_cast<const uint32_t*>(ws + W.ready);
    const int H = d.H, R = kSeg ? seg->ntasks : d.N * d.H;
    volatile int* abort = &sm.abort;

    if (tid == 0) {
        ptx::mbar_init(&sm.wq_full, 1);
        ptx::mbar_init(&sm.kt_full, 1);
        ptx::mbar_init(&sm.u_full, 1);
        ptx::mbar_init(&sm.p_full[0], 1);
        ptx::mbar_init(&sm.p_full[1], 1);
        ptx::mbar_init(&sm.d1, 2);  // the two halves of (w S)^T
        ptx::mbar_init(&sm.d2, 1);
        ptx::mbar_init(&sm.d3[0], 1);
        ptx::mbar_init(&sm.d3[1], 1);
        ptx::mbar_init(&sm.fin, 3);  // the three issuing threads
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    auto chain_at = [&](int r) {
        ChainPos p{r, 0, 0, 0, 0, 0, 0, 0, kTaskWhole};
        if (kSeg) {
            if (r < R) {
                const int4 t = seg->tasks[r];
                p.c0 = t.x;
                p.len = t.y;
                p.s = t.z / H;
                p.h = t.z - p.s * H;
                p.w = t.w;
                if (p.len > 0) {
                    p.tok0 = chunk_tab[p.c0].y;
                    p.ntok = kChunk * (p.len - 1) + chunk_tab[p.c0 + p.len - 1].z;
                }
            }
            return p;
        }
        if (r < R) {
            p.h = r % H;
            p.s = order[r / H];
            p.c0 = seq_first[p.s];
            p.len = seq_first[p.s + 1] - p.c0;
            if (p.len > 0) {
                p.tok0 = chunk_tab[p.c0].y;
                p.ntok = kChunk * (p.len - 1) + chunk_tab[p.c0 + p.len - 1].z;
            }
        }
        return p;
    };
    // The step after p in this CTA's list, or one with len == 0 (none: chains are
    // ranked longest first, so once one is empty so are all later ones).
    auto next_of = [&](ChainPos p) {
        if (p.j + 1 < p.len) {
            ++p.j;
            return p;
        }
        return chain_at(p.r + nc);
    };
    auto block_of = [&](const ChainPos& p) {
        return ws + W.factors + ((size_t)(p.c0 + p.j) * H + p.h) * W.factor_bytes;
    };
    auto flag_of = [&](const ChainPos& p) { return ready + (size_t)(p.c0 + p.j) * H + p.h; };
    // The copy thread (lane 0 of warp 2) acquires the ready flags and issues every
    // bulk copy; threads 0 and 32 issue the serial part of GEMM1 (thread 0 also
    // GEMM2), thread 96 its output part and GEMM3.  Copies are counted so that a CTA
    // that leaves early can wait for those still in flight.
    constexpr int kCopier = 64;
    uint32_t n_wq = 0, n_kt = 0, n_u = 0, n_p0 = 0, n_p1 = 0;
    auto issue_wq = [&](const ChainPos& p) {
        ptx::mbar_arrive_expect_tx(&sm.wq_full, WQB);
        ptx::bulk_g2s(sm.WQ, block_of(p) + F.wq, WQB, &sm.wq_full);
        ++n_wq;
    };
    auto issue_u = [&](const ChainPos& p) {
        ptx::mbar_arrive_expect_tx(&sm.u_full, UB);
        ptx::bulk_g2s(sm.U0, block_of(p) + F.u0, UB, &sm.u_full);
        ++n_u;
    };
    auto issue_kt = [&](const ChainPos& p, int slot) {
        ptx::mbar_arrive_expect_tx(&sm.kt_full, KTB + GLB);
        ptx::bulk_g2s(sm.KT, block_of(p) + F.kt, KTB, &sm.kt_full);
        ptx::bulk_g2s(sm.GL[slot], block_of(p) + F.gl, GLB, &sm.kt_full);
        ++n_kt;
    };
    auto issue_p = [&](const ChainPos& p, int slot) {
        ptx::mbar_arrive_expect_tx(&sm.p_full[slot], PB);
        ptx::bulk_g2s(sm.P[slot], block_of(p) + F.p, PB, &sm.p_full[slot]);
        ++(slot ? n_p1 : n_p0);
    };
    // Flags are acquired in batches: relaxed loads of up to kLook steps' flags side
    // by side, then one acquire fence for the published prefix, so that the flag
    // latency is paid about once per batch while the producers run ahead.
    constexpr int kLook = 8;
    uint32_t ready_to = 0;  // (copy thread) steps below this one are acquired
    auto acquire = [&](uint32_t step, const ChainPos& p0) -> bool {  // p0: the position of `step`
        if (step < ready_to || !use_flags) return true;
        ChainPos p = p0;
        uint32_t v[kLook];
        int nl = 0;
#pragma unroll
        for (int k2 = 0; k2 < kLook; ++k2) {
            v[k2] = 0;
            if (p.len > 0 && nl == k2) {
                v[k2] = ptx::ld_relaxed_gpu(flag_of(p));
                ++nl;
                p = next_of(p);
            }
        }
        int got = 0;
#pragma unroll
        for (int k2 = 0; k2 < kLook; ++k2)
            if (got == k2 && k2 < nl && v[k2] != 0) ++got;
        if (got == 0) {  // the first is not out yet
            if (!ptx::flag_spin(flag_of(p0), err, abort)) return false;
            got = 1;
        }
        ptx::fence_acquire_for_bulk();
        ready_to = step + (uint32_t)got;
        return true;
    };

    ChainPos cur = chain_at((int)blockIdx.x);
    bool have = cur.len > 0;
    bool copies_ok = true;  // (copy thread) every flag so far acquired
    if (tid == kCopier && have) {
        if (acquire(0, cur)) {
            issue_wq(cur);
            issue_u(cur);
            issue_kt(cur, 0);
            issue_p(cur, 0);
        } else {
            copies_ok = false;
            chain_raise(ws, abort);
        }
    }
    bool ok = true;
    float S[32];  // S^T: value column n, channels 32 g .. 32 g + 31
#pragma unroll
    for (int e = 0; e < 32; ++e) S[e] = 0.f;
    bool have_prev = false;
    int4 prev_out = make_int4(0, 0, 0, 0);  // {first token row, rows, head, 0} of the previous step
    ChainPos prev_pos = cur;                // the previous step
    // The previous step's factor block: every part of it has been read (its GEMM3,
    // the last reader, is done) and nothing else reads it, so its lines leave L2
    // without being written back.
    auto drop_prev_block = [&]() {
        if (kSeg && !task_outputs(prev_pos.w)) return;  // a map task: the tail task reads it again
        const uint8_t* blk = block_of(prev_pos);
        for (int i = tid; i < (int)(W.factor_bytes / 128); i += kThreads) ptx::discard_l2_line(blk + 128 * i);
    };
    uint32_t gj = 0;                        // steps of this CTA so far
    // The output leaves in two moves: each thread puts its 16 rows of column n from
    // tensor memory into a row-major staging tile; after the next barrier, lane 0 of
    // warps 4-15 sends the tile's valid rows out with one bulk copy each (so that no
    // thread's load/store pipe holds synchronous stores on the chain's critical path).
    TOut* const otile = reinterpret_cast<TOut*>(sm.otile);
    int4 tile_out = make_int4(0, 0, 0, 0);  // {first token row, rows, head, staged?} of the tile
    auto out_stage = [&](uint32_t buf) {    // output of the step in D1^T[buf]: rows 16 g ..
        float acc[16];
        ptx::tmem_ld16(tmem + lb + kTO + 64 * buf + 16 * g, acc);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) store_out(otile + (16 * g + i) * DV + n, scale * acc[i]);
        ptx::fence_proxy_async_smem();  // the bulk copies read the tile
        tile_out = make_int4(prev_out.x, prev_out.y, prev_out.z, 1);
    };
    auto out_flush = [&]() {  // issue the row copies (the tile's reads end before the next barrier)
        if (tile_out.w && warp >= 4 && lane == 0) {
            for (int row = warp - 4; row < tile_out.y; row += 12)
                ptx::bulk_s2g(o + ((size_t)(tile_out.x + row) * H + tile_out.z) * DV, otile + row * DV,
                              DV * (uint32_t)sizeof(TOut));
            ptx::bulk_commit();
        }
        tile_out.w = 0;
    };
    auto out_flush_wait = [&]() {  // the tile may be written again
        if (warp >= 4 && lane == 0) ptx::bulk_wait_read_all();
    };
    while (have && ok) {
        const ChainPos nxt = next_of(cur);
        const bool nv = nxt.len > 0;
        const uint32_t b = gj & 1u;
        // -------- a new chain: its initial state into S^T and the bf16 copy
        if (cur.j == 0) {
            const size_t base = ((size_t)cur.s * H + cur.h) * DK * DV;
            const float* src = h0 ? h0 + base : nullptr;
            bool ident = false;
            if (kSeg) {
                const int kind = cur.w & 7;
                if (kind == kTaskMapF || kind == kTaskMapZ) src = nullptr;
                if (kind == kTaskMapF) ident = true;
                if (kind == kTaskTail) src = seg->E + (size_t)(cur.w >> 4) * DK * DV;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e)
                S[e] = ident ? (32 * g + e == n ? 1.f : 0.f) : src ? src[(size_t)(32 * g + e) * DV + n] : 0.f;
            uint32_t sb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sb[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
            ptx::tmem_st16(tmem + lb + kTS + 16 * g, sb);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ok = __syncthreads_and(ok && !*abort);
            if (!ok) break;
        }
        // -------- GEMM1, the part on the serial path: (w S)^T = S^T w^T, its two
        //          halves over the channels issued side by side (threads 0 and 32)
        if (tid == 0 || tid == 32) {
            if (ptx::mbar_spin_or_abort(&sm.wq_full, b, abort)) {
                ptx::tc_fence_after();
                constexpr uint32_t idw = ptx::idesc_bf16(128, kChunk) | kBMajorMN;
                const uint64_t bd = ptx::smem_desc(ptx::smem_u32(sm.WQ), 128, (DK / 8) * 128);
                const int k0 = tid == 0 ? 0 : DK / 32;
#pragma unroll
                for (int kk = 0; kk < DK / 32; ++kk)
                    ptx::mma_bf16_ta(tmem + (tid == 0 ? kTXa : kTXb), tmem + kTS + 8 * (k0 + kk),
                                     bd + (uint64_t)(((k0 + kk) * 256) >> 4), idw, kk > 0);
                ptx::mma_commit(&sm.d1);
            } else {
                chain_raise(ws, abort);
            }
        } else if (tid == 96) {
            // GEMM1, the output part: O^T[b] = S^T QG^T (its B: rows 64-127 of [w; QG]);
            // issued beside the serial part (the thread would wait for d1 meanwhile)
            if (ptx::mbar_spin_or_abort(&sm.wq_full, b, abort)) {
                ptx::tc_fence_after();
                constexpr uint32_t idq = ptx::idesc_bf16(128, kChunk) | kBMajorMN;
                const uint64_t bd = ptx::smem_desc(ptx::smem_u32(sm.WQ) + kChunk * DK * 2, 128, (DK / 8) * 128);
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk)
                    ptx::mma_bf16_ta(tmem + kTO + 64 * b, tmem + kTS + 8 * kk, bd + (uint64_t)((kk * 256) >> 4),
                                     idq, kk > 0);
            } else {
                chain_raise(ws, abort);
            }
        }
        // -------- U^T = u^T - (w S)^T (the previous GEMM3, the last reader of the
        //          bf16 U^T, is done first)
        out_flush();  // the tile staged last step (the barrier after it has passed)
        bool okl = gj == 0 || ptx::mbar_spin_or_abort(&sm.d3[(gj - 1) & 1u], ((gj - 1) >> 1) & 1u, abort);
        okl = okl && ptx::mbar_spin_or_abort(&sm.d1, b, abort);
        okl = okl && ptx::mbar_spin_or_abort(&sm.u_full, b, abort);
        okl = __all_sync(0xffffffffu, okl);
        if (okl) {
            ptx::tc_fence_after();
            float4 un[4];  // u: value column n, rows 16 g .. 16 g + 15
            const float4* u0 = reinterpret_cast<const float4*>(sm.U0) + 4 * g * DV + n;
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) un[k2] = u0[k2 * DV];
            float uu[16];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {
                uu[4 * k2] = un[k2].x; uu[4 * k2 + 1] = un[k2].y; uu[4 * k2 + 2] = un[k2].z; uu[4 * k2 + 3] = un[k2].w;
            }
            if (kSeg && (cur.w & 7) == kTaskMapF) {  // the map: the step without its u
#pragma unroll
                for (int e = 0; e < 16; ++e) uu[e] = 0.f;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // minus both halves of (w S)^T
                float acc[16];
                ptx::tmem_ld16(tmem + lb + (half ? kTXb : kTXa) + 16 * g, acc);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) uu[e] -= acc[e];
            }
            uint32_t ut[16], ub[8];
#pragma unroll
            for (int e = 0; e < 16; ++e) ut[e] = __float_as_uint(uu[e]);
#pragma unroll
            for (int i = 0; i < 8; ++i) ub[i] = pack_bf16(__uint_as_float(ut[2 * i]), __uint_as_float(ut[2 * i + 1]));
            ptx::tmem_st16(tmem + lb + kTXa + 16 * g, ut);
            ptx::tmem_st8(tmem + lb + kTUB + 8 * g, ub);
            ptx::tmem_st_wait();
        }
        out_flush_wait();
        if (tid == kCopier && okl && nv && copies_ok) {
            // next step: its flag, then P (slot b^1, read by the previous GEMM3) and
            // [w; QG] (read by this GEMM1)
            copies_ok = acquire(gj + 1, nxt);
            if (copies_ok) {
                issue_p(nxt, (int)(b ^ 1u));
                issue_wq(nxt);
            } else {
                chain_raise(ws, abort);
            }
        }
        ptx::tc_fence_before();
        ok = __syncthreads_and(ok && okl);
        if (!ok) break;
        // -------- GEMM2: D2^T = U^T KT^T (tf32, the serial path); GEMM3: O^T += U^T P^T
        if (tid == kCopier && nv && copies_ok) issue_u(nxt);  // u has been read
        if (tid == 0) {
            if (ptx::mbar_spin_or_abort(&sm.kt_full, b, abort)) {
                ptx::tc_fence_after();
                constexpr uint32_t id2 = ptx::idesc_tf32(128, DK);
                const uint64_t bd = ptx::smem_desc(ptx::smem_u32(sm.KT), (DK / 8) * 128, 128);
#pragma unroll
                for (int kk = 0; kk < kChunk / 8; ++kk)
                    ptx::mma_tf32_ta(tmem + kTD2, tmem + kTXa + 8 * kk,
                                     bd + (uint64_t)((kk * 2 * (DK / 8) * 128) >> 4), id2, kk > 0);
                ptx::mma_commit(&sm.d2);
            } else {
                chain_raise(ws, abort);
            }
        } else if (tid == 96) {
            if (ptx::mbar_spin_or_abort(&sm.p_full[b], (gj >> 1) & 1u, abort)) {
                ptx::tc_fence_after();
                constexpr uint32_t id3 = ptx::idesc_bf16(128, kChunk);
                const uint64_t bd = ptx::smem_desc(ptx::smem_u32(sm.P[b]), 1024, 128);
#pragma unroll
                for (int kk = 0; kk < kChunk / 16; ++kk)
                    ptx::mma_bf16_ta(tmem + kTO + 64 * b, tmem + kTUB + 8 * kk,
                                     bd + (uint64_t)((kk * 2048) >> 4), id3, true);
                ptx::mma_commit(&sm.d3[b]);
            } else {
                chain_raise(ws, abort);
            }
        }
        // -------- output of the previous step into the staging tile, and its factor
        //          block out of L2 (its GEMM3 was waited for before the barrier), while
        //          GEMM2 runs
        if (have_prev && (!kSeg || task_outputs(prev_pos.w))) {
            ptx::tc_fence_after();
            out_stage(b ^ 1u);
            drop_prev_block();
        }
        // -------- S^T <- S^T Diag(GL) + D2^T  ->  bf16 S^T (GEMM1, its reader, is done)
        bool okd = ptx::mbar_spin_or_abort(&sm.d2, b, abort);
        okd = __all_sync(0xffffffffu, okd);
        if (tid == kCopier && okd && nv && copies_ok) issue_kt(nxt, (int)(b ^ 1u));  // GEMM2 has read KT
        if (okd) {
            ptx::tc_fence_after();
            float acc[32];
            ptx::tmem_ld16(tmem + lb + kTD2 + 32 * g, *reinterpret_cast<float(*)[16]>(&acc[0]));
            ptx::tmem_ld16(tmem + lb + kTD2 + 32 * g + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
            ptx::tmem_ld_wait();
            const float4* gl4 = reinterpret_cast<const float4*>(sm.GL[b] + 32 * g);
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
                const float4 gv = gl4[k2];
                S[4 * k2] = fmaf(gv.x, S[4 * k2], acc[4 * k2]);
                S[4 * k2 + 1] = fmaf(gv.y, S[4 * k2 + 1], acc[4 * k2 + 1]);
                S[4 * k2 + 2] = fmaf(gv.z, S[4 * k2 + 2], acc[4 * k2 + 2]);
                S[4 * k2 + 3] = fmaf(gv.w, S[4 * k2 + 3], acc[4 * k2 + 3]);
            }
            uint32_t sb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sb[i] = pack_bf16(S[2 * i], S[2 * i + 1]);
            ptx::tmem_st16(tmem + lb + kTS + 16 * g, sb);
            ptx::tmem_st_wait();
            if (cur.j == cur.len - 1) {  // the chain's last chunk: its final state
                float* dst = hT ? hT + ((size_t)cur.s * H + cur.h) * DK * DV : nullptr;
                if (kSeg) {
                    const int kind = cur.w & 7;
                    const size_t slot = (size_t)(cur.w >> 4) * DK * DV;
                    if (kind == kTaskHead || kind == kTaskMapZ) dst = seg->E + slot;
                    if (kind == kTaskTail && !((cur.w >> 3) & 1)) dst = nullptr;  // the scan made it
                    if (kind == kTaskMapF) {  // the map, transposed: F^T[n][c] (padded rows), 32 floats per thread
                        constexpr int LD = DK + kMapPad;
                        float4* ft = reinterpret_cast<float4*>(seg->F + (size_t)(cur.w >> 4) * DK * LD +
                                                               (size_t)n * LD + 32 * g);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            ft[e] = make_float4(S[4 * e], S[4 * e + 1], S[4 * e + 2], S[4 * e + 3]);
                        dst = nullptr;
                    }
                }
                if (dst) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[(size_t)(32 * g + e) * DV + n] = S[e];
                }
            }
        }
        ptx::tc_fence_before();
        ok = __syncthreads_and(ok && okd);
        {
            const int rows = cur.ntok - kChunk * cur.j;
            prev_out = make_int4(cur.tok0 + kChunk * cur.j, rows < kChunk ? rows : kChunk, cur.h, 0);
        }
        have_prev = true;
        prev_pos = cur;
        ++gj;
        cur = nxt;
        have = nv;
    }
    // -------- the last step's output (ok and have_prev are the same in every thread)
    if (ok && have_prev) {
        out_flush();
        out_flush_wait();
        bool okl = ptx::mbar_wait_or_abort(&sm.d3[(gj - 1) & 1u], ((gj - 1) >> 1) & 1u, abort);
        okl = __all_sync(0xffffffffu, okl);
        ok = __syncthreads_and(okl);  // the tile is free again
        if (ok) {
            ptx::tc_fence_after();
            if (!kSeg || task_outputs(prev_pos.w)) {
                out_stage((gj - 1) & 1u);
                drop_prev_block();
            }
        } else {
            chain_raise(ws, abort);
        }
        __syncthreads();
        if (ok) out_flush();
    }
    if (warp >= 4 && lane == 0) ptx::bulk_wait_all();  // the output rows have left
    // -------- empty chains (zero-length sequences): the state passes through
    if (hT) {
        for (int r = (int)blockIdx.x; r < R; r += nc) {
            const ChainPos p = chain_at(r);
            if (p.len > 0) continue;
            const size_t base = ((size_t)p.s * H + p.h) * DK * DV;
            for (int e = tid; e < DK * DV; e += kThreads) hT[base + e] = h0 ? h0[base + e] : 0.f;
        }
    }
    // -------- leave cleanly: copies in flight land, issued MMAs complete, TMEM goes
    {
        volatile int never = 0;
        if (tid == kCopier) {
            if (n_wq) ptx::mbar_wait_or_abort(&sm.wq_full, (n_wq - 1) & 1u, &never);
            if (n_kt) ptx::mbar_wait_or_abort(&sm.kt_full, (n_kt - 1) & 1u, &never);
            if (n_u) ptx::mbar_wait_or_abort(&sm.u_full, (n_u - 1) & 1u, &never);
            if (n_p0) ptx::mbar_wait_or_abort(&sm.p_full[0], (n_p0 - 1) & 1u, &never);
            if (n_p1) ptx::mbar_wait_or_abort(&sm.p_full[1], (n_p1 - 1) & 1u, &never);
        }
        if (tid == 0 || tid == 32 || tid == 96) ptx::mma_commit(&sm.fin);
        if (tid == 0) ptx::mbar_wait_or_abort(&sm.fin, 0, &never);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// The first n_chain CTAs (Header::n_chain, set by the schedule kernel) run chains;
// the others produce factors, positions (blockIdx - n_chain) + n (grid - n_chain) of
// the production order, with u in the transposed layout the chains read.
template <typename TIn, typename TG>
__global__ void __launch_bounds__(kThreads, 1)
    fused_kernel(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                 const float* __restrict__ beta, const float* __restrict__ h0, float scale,
                 TIn* __restrict__ o, float* __restrict__ hT, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const WsLayout W(d);
    const int nc = reinterpret_cast<const Header*>(ws + W.header)->n_chain;
    if (nc <= 0) return;  // malformed cu_seqlens (reported in the error word): nothing to do
    if ((int)blockIdx.x < nc) {
        chain_role<TIn>(d, h0, scale, o, hT, ws, smem_raw, nc, true);
    } else {
        const ItemPlan plan{reinterpret_cast<const int32_t*>(ws + W.plist), (int)blockIdx.x - nc,
                            (int)gridDim.x - nc, reinterpret_cast<uint32_t*>(ws + W.ready), true};
        factor_body<kCDK, kCDV, TIn, TG>(d, &tm_q, &tm_k, &tm_v, &tm_g, beta, ws, smem_raw, plan);
    }
}

// The split pipeline's 128-column chain kernel: the fused kernel's chain role over
// factor blocks that the factor kernel has finished; runs only when the schedule
// kernel chose it for these chain lengths.
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    chain128_kernel(Dims d, const float* __restrict__ h0, float scale, TIn* __restrict__ o,
                    float* __restrict__ hT, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const WsLayout W(d);
    if (!reinterpret_cast<const Header*>(ws + W.header)->chain128) return;
    chain_role<TIn>(d, h0, scale, o, hT, ws, smem_raw, (int)gridDim.x, false);
}

template <typename TIn>
cudaError_t launch_chain128_t(const Dims& d, const float* h0, float scale, void* o, float* hT, uint8_t* ws,
                              cudaStream_t stream) {
    auto kern = chain128_kernel<TIn>;
    const size_t smem = sizeof(ChainRoleSmem);
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const long long chains = (long long)d.N * d.H;
    if (chains == 0) return cudaSuccess;
    const unsigned grid = (unsigned)(chains < num_sms() ? chains : num_sms());
    kern<<<grid, kThreads, smem, stream>>>(d, h0, scale, static_cast<TIn*>(o), hT, ws);
    return cudaGetLastError();
}

// A pass of segmented chains (the split pipeline for few long chains): pass 0 runs
// the first segments from h0 and the middle segments' maps F and states from zero Z;
// pass 1 the segments after the first from the start states the scan made.  Each
// task is a chain of the chain role; runs only when the schedule kernel chose
// segments.
template <typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    seg_chain_kernel(Dims d, const float* __restrict__ h0, float scale, TIn* __restrict__ o,
                     float* __restrict__ hT, uint8_t* __restrict__ ws, int pass) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const WsLayout W(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    if (!hdr->seg) return;
    const SegRun run{reinterpret_cast<const int4*>(ws + (pass ? W.seg_c : W.seg_a)),
                     pass ? hdr->seg_nc : hdr->seg_na, reinterpret_cast<float*>(ws + W.seg_e),
                     reinterpret_cast<float*>(ws + W.seg_f)};
    chain_role<TIn, true>(d, h0, scale, o, hT, ws, smem_raw, (int)gridDim.x, false, &run);
}

template <typename TIn>
cudaError_t launch_seg_pass_t(const Dims& d, int pass, const float* h0, float scale, void* o, float* hT,
                              uint8_t* ws, cudaStream_t stream) {
    auto kern = seg_chain_kernel<TIn>;
    const size_t smem = sizeof(ChainRoleSmem);
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const int sms = num_sms();
    const unsigned grid = (unsigned)(sms < kSegTasks ? sms : kSegTasks);
    kern<<<grid, kThreads, smem, stream>>>(d, h0, scale, static_cast<TIn*>(o), hT, ws, pass);
    return cudaGetLastError();
}

template <typename TIn>
constexpr size_t fused_smem() {
    return sizeof(FactorSmem<kCDK, kCDV, TIn>) > sizeof(ChainRoleSmem) ? sizeof(FactorSmem<kCDK, kCDV, TIn>)
                                                                       : sizeof(ChainRoleSmem);
}

template <typename TIn, typename TG>
cudaError_t launch_fused_t(const Dims& d, const void* q, const void* k, const void* v, const void* g,
                           const float* beta, const float* h0, float scale, void* o, float* hT, uint8_t* ws,
                           cudaStream_t stream) {
    static_assert(fused_smem<TIn>() <= 227 * 1024, "fused kernel shared memory");
    constexpr int DK = kCDK, DV = kCDV;
    auto kern = fused_kernel<TIn, TG>;
    const size_t smem = fused_smem<TIn>();
    const long long tokens = (long long)d.B * d.T;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    constexpr bool f32 = sizeof(TIn) == 4;
    // With no token at all (the inputs may then be null) the maps describe 64 rows
    // at the workspace instead; no item exists, so they are never used.
    const bool none = tokens == 0;
    const long long rows = none ? kChunk : tokens;
    const void *bq = none ? ws : q, *bk = none ? ws : k, *bv = none ? ws : v, *bg = none ? ws : g;
    CUtensorMap tq, tk, tv, tg;
    const bool okv = f32 ? encode_rows(&tv, bv, true, DV, d.H, rows) : encode_groups(&tv, bv, DV, d.H, rows);
    if (!encode_rows(&tq, bq, f32, DK, d.H, rows) || !encode_rows(&tk, bk, f32, DK, d.H, rows) || !okv ||
        !encode_rows(&tg, bg, sizeof(TG) == 4, DK, d.H, rows))
        return cudaErrorInvalidValue;
    const int grid = fused_grid(d);
    if (grid < 2) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // chain CTAs wait for factor CTAs
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, d, tq, tk, tv, tg, beta, h0, scale, static_cast<TIn*>(o), hT, ws);
}

}  // namespace

int fused_grid(const Dims& d) {
    const int sms = num_sms();
    if (d.dk != kCDK || d.dv != kCDV || sms < 2 || sms > 1025 || d.N > kRankMax || (long long)d.N * d.H > 65536)
        return 0;
    return sms;
}

// One item's factors take about this many chain steps (measured on GB300 with bf16
// inputs: about 9.5 us per item on a factor CTA, 2.4 us per chain step).
float fused_ratio(const Dims& d, bool qkv_bf16) {
    (void)d;
    return qkv_bf16 ? 4.f : 5.f;
}

bool chain128_applies(const Dims& d) { return d.dk == kCDK && d.dv == kCDV && d.N <= kRankMax; }

cudaError_t launch_chain128(const Dims& d, bool qkv_bf16, const float* h0, float scale, void* o,
                            float* hT, uint8_t* ws, cudaStream_t stream) {
    if (!chain128_applies(d)) return cudaErrorInvalidValue;
    return qkv_bf16 ? launch_chain128_t<__nv_bfloat16>(d, h0, scale, o, hT, ws, stream)
                    : launch_chain128_t<float>(d, h0, scale, o, hT, ws, stream);
}

cudaError_t launch_seg_pass(const Dims& d, bool qkv_bf16, int pass, const float* h0, float scale,
                            void* o, float* hT, uint8_t* ws, cudaStream_t stream) {
    if (!seg_layout_applies(d)) return cudaErrorInvalidValue;
    return qkv_bf16 ? launch_seg_pass_t<__nv_bfloat16>(d, pass, h0, scale, o, hT, ws, stream)
                    : launch_seg_pass_t<float>(d, pass, h0, scale, o, hT, ws, stream);
}

cudaError_t launch_fused(const Dims& d, bool qkv_bf16, bool g_bf16, const void* q, const void* k,
                         const void* v, const void* g, const float* beta, const float* h0,
                         float scale, void* o, float* hT, uint8_t* ws, cudaStream_t stream) {
    using bf = __nv_bfloat16;
    if (d.dk != kCDK || d.dv != kCDV) return cudaErrorInvalidValue;
    if (!qkv_bf16)
        return g_bf16 ? cudaErrorInvalidValue
                      : launch_fused_t<float, float>(d, q, k, v, g, beta, h0, scale, o, hT, ws, stream);
    return g_bf16 ? launch_fused_t<bf, bf>(d, q, k, v, g, beta, h0, scale, o, hT, ws, stream)
                  : launch_fused_t<bf, float>(d, q, k, v, g, beta, h0, scale, o, hT, ws, stream);
}

}  // namespace kda
