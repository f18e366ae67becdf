#pragma once
// Per-chunk factors of the chunkwise KDA forward, every chunk product on tcgen05:
// the body of a persistent 512-thread CTA (one per SM) that walks (chunk, head)
// items in a given order (ItemPlan: head-major in the factor kernel, the
// production order in the fused kernel).  The next item's q, k, g arrive by TMA
// tensor copies while the current item is still in its products, its v tile lands
// straight in the tensor-core operand layout, and every result leaves by coalesced
// 16-byte stores from registers (phases P1-P7 below).
//
// For a chunk of L <= 64 tokens of one sequence and head ("Autoresearch on Kimi
// Delta Attention", section THE MECHANISM: inside a block the work becomes matrix
// products; "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 03
// REWARD HACKING: L2 normalisation of q and k, the cumulative decay inside each
// 64-token chunk, the triangular inverse):
//   qh, kh   = rows of q, k over sqrt(|x|^2 + eps)                  (fp32)
//   alpha    = exp(g)                                              (one exp per element)
//   A_ij     = beta_i sum_c kh_ic kh_jc D_c(i, j)                     j < i
//   P_ij     = sum_c qh_ic kh_jc D_c(i, j)                            j <= i
//   with D_c(i, j) = exp(Gamma_ic - Gamma_jc) = alpha_c(j+1) ... alpha_c(i)
//   X        = (I + A)^-1                                           (fp32, blocked)
//   u        = X Diag(beta) v                                        (tcgen05, M=64 N=dv K=64)
//   w^T      = (kh * gamma)^T (X Diag(beta))^T                       (tcgen05, M=dk N=64 K=64)
//   QG = qh * gamma,  KT = (kh * gamma_L / gamma)^T,  GL = gamma_L,  gamma = exp(Gamma)
// X Diag(beta) enters both products split into bf16 hi + lo (two MMA passes).
//
// Decay factors without overflow.  Every decay factor is a product of alphas over
// a run of consecutive tokens, so it lies in [0, 1]: deep decays underflow to zero
// and nothing overflows (the pages' section 03 describes kernels that formed
// exp(Gamma) / exp(Gamma') and produced NaN).  A and P are split by levels: a pair
// (i, j), j < i, belongs to the level s = 2^l of the highest bit in which i and j
// differ, so that inside an aligned block of 2s rows i lies in the upper half and j
// in the lower, and the half boundary m separates them.  With m as reference,
//   D(i, j) = D(i, m) D(m, j),   D(i, m) = alpha(m+1 .. i),   D(m, j) = alpha(j+1 .. m),
// both in [0, 1], so every level is one plain matrix product of row-scaled and
// column-scaled keys.  The six levels (s = 1 .. 32) each hold 32 rows and 32
// columns; two levels share one M = 128, N = 64 tensor-core product (rows
// [kh R; qh R] of both levels, columns kh C of both), whose two diagonal 32 x 32
// blocks are the wanted results and whose off-diagonal blocks are ignored.
#include <cuda.h>          // CUtensorMap (the encoder itself is fetched at run time)
#include <cudaTypedefs.h>  // the encoder's function-pointer type

#include <type_traits>

#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

// Tensor maps of the inputs (defined in kda_factor.cu).
bool encode_rows(CUtensorMap* m, const void* base, bool f32, int D, int H, long long tokens);
bool encode_groups(CUtensorMap* m, const void* base, int D, int H, long long tokens);

// The items one factor CTA produces: positions first, first + stride, ... of an
// order of the (chunk, head) items.  list: the order as chunk * H + head per
// position, or nullptr for head-major (position h * total + c).  ready: flags set
// (release, GPU scope) once an item's factor block is complete in global memory,
// or nullptr.
struct ItemPlan {
    const int32_t* list;
    int first, stride;
    uint32_t* ready;
    bool ut;  // u leaves as [64/4][dv][4] (the 128-column chains' layout), else slabbed
};

namespace {

constexpr int kThreads = 512;
constexpr int kIssuer2 = 256;  // the second tensor-core issuing thread (lane 0 of warp 8)
constexpr int kIssuer3 = 384;  // the third (lane 0 of warp 12)
constexpr uint32_t kAMajorMN = 1u << 15;  // instruction-descriptor bit: A is M-major
constexpr uint32_t kBMajorMN = 1u << 16;  // instruction-descriptor bit: B is N-major
constexpr int AP = kChunk + 1;            // row stride of the fp32 A and X arrays

// Once the level products are done, the operand ring holds the inverse's arrays.
constexpr int kOffA = 0;                              // A (fp32, 64 x 65)
constexpr int kOffX = kChunk * AP * 4;                // X (fp32, 64 x 65)
constexpr int kOffScr = 2 * kChunk * AP * 4;          // inverse scratch (32 x 32 fp32)
constexpr int kOffPst = kOffScr + 32 * 32 * 4;        // P staging (fp32, 64 x 65)
constexpr int kInvBytes = kOffPst + kChunk * AP * 4;
constexpr int kOffXop = 0;                            // X Diag(beta), bf16 hi (over A)
constexpr int kOffXlo = kChunk * kChunk * 2;          // and its remainder lo

template <int DK, int DV, typename TIn>
struct FactorCfg {
    static constexpr int NBUF = sizeof(TIn) == 2 ? 2 : 1;  // level operand buffers
    static constexpr int PAIR = 128 * DK * 2 + 64 * DK * 2; // [kh R; qh R] x 2 levels + kh C x 2
    static constexpr int RING0 = NBUF * PAIR > kInvBytes ? NBUF * PAIR : kInvBytes;
    // fp32 inputs: the fp32 v tile also lands in the ring before it is converted
    static constexpr int RING1 = (sizeof(TIn) == 4 && kChunk * DV * 4 > RING0) ? kChunk * DV * 4 : RING0;
    static constexpr int RING = (RING1 + 1023) / 1024 * 1024;
};

template <int DK, int DV, typename TIn>
struct __align__(1024) FactorSmem {
    using C = FactorCfg<DK, DV, TIn>;
    uint8_t ring[C::RING];               // level operands, then A, X, X Diag(beta) hi/lo
    TIn qr[kChunk * DK];                 // raw q rows as copied in; qh = qr * iq[row]
    TIn kr[kChunk * DK];                 // raw k rows; kh = kr * ik[row]
    float gr[kChunk * DK];               // raw g rows as copied in (fp32, or bf16 in the first half)
    // v: bf16 inputs, the N-major bf16 operand [DV/8][64 rows][8 columns]; fp32
    // inputs, the K-major tf32 operand (DV x 64, 4 chunk rows per 16-byte core row)
    std::conditional_t<sizeof(TIn) == 2, __nv_bfloat16, float> vs[kChunk * DV];
    // (kh * gamma)^T, K-major bf16 operand (DK x 64); with fp32 inputs it is a tf32
    // operand in the q staging, dead by then, and this array is unused
    __nv_bfloat16 kg[sizeof(TIn) == 2 ? DK * kChunk : 8];
    float blk_a[8 * DK];                 // alpha at the first row of each 8-row block
    float blk_t[8 * DK];                 // product of alpha over rows 1..7 of each block
    float diag[2 * kChunk];              // qh_i . kh_i, one partial sum per channel half
    float bs[2][kChunk];                 // beta (zero past the chunk end), alternate items
    float iq[kChunk], ik[kChunk];        // inverse row norms (zero past the chunk end)
    uint64_t ld_bar, v_bar, lv_bar[3], wu_bar, drain_bar;
    uint32_t tmem;
    int abort;
};

// Byte offset of (rank m, channel c) in an M-major (MN-major) operand with K = DK:
// core matrices of 8 channels (16-byte rows of 8 consecutive ranks), channel-
// adjacent cores 128 B apart (descriptor leading byte offset 128), rank-adjacent
// cores DK/8 * 128 B apart (stride byte offset).
template <int DK>
__device__ __forceinline__ uint32_t mn_off(int m, int c) {
    return (uint32_t)((((m >> 3) * (DK >> 3) + (c >> 3)) << 7) + ((c & 7) << 4) + ((m & 7) << 1));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
}

// Four values (ranks m .. m+3, m % 4 == 0) or eight (m % 8 == 0) of one channel.
template <int DK>
__device__ __forceinline__ void st4(uint8_t* base, int m, int c, float a, float b, float x, float y) {
    *reinterpret_cast<uint2*>(base + mn_off<DK>(m, c)) = make_uint2(pack_bf16(a, b), pack_bf16(x, y));
}
template <int DK>
__device__ __forceinline__ void st8(uint8_t* base, int m, int c, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(base + mn_off<DK>(m, c)) = pack8(v);
}

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

// 8 elements from 16-byte words: one word of bf16, or two of fp32.
template <typename T>
__device__ __forceinline__ void unpack8(const uint4* w, float (&x)[8]);
template <>
__device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4* w, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
template <>
__device__ __forceinline__ void unpack8<float>(const uint4* w, float (&x)[8]) {
    const float* f = reinterpret_cast<const float*>(w);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = f[i];
}

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma1688_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// C (16 x 8 tile at rows cr, cols cc of an N x N block, row stride ldc) = P Q over
// K = N, P and Q read from fp32 shared memory (row strides ldp, ldq), tf32 inputs,
// fp32 accumulation; sign -1 negates.  One warp.  LOWER_P / LOWER_Q: that operand
// is lower triangular and its strict upper triangle, never written, reads as zero.
template <int N, bool LOWER_P, bool LOWER_Q>
__device__ __forceinline__ void tile_mm_tf32(const float* P, int ldp, const float* Q, int ldq,
                                             float* C, int ldc, int cr, int cc, float sign,
                                             int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    auto pv = [&](int r, int k) { return (LOWER_P && k > r) ? 0.f : P[r * ldp + k]; };
    auto qv = [&](int k, int n) { return (LOWER_Q && n > k) ? 0.f : Q[k * ldq + n]; };
#pragma unroll
    for (int k0 = 0; k0 < N; k0 += 8) {
        uint32_t a[4];
        a[0] = to_tf32(pv(cr + gq, k0 + tq));
        a[1] = to_tf32(pv(cr + gq + 8, k0 + tq));
        a[2] = to_tf32(pv(cr + gq, k0 + tq + 4));
        a[3] = to_tf32(pv(cr + gq + 8, k0 + tq + 4));
        const uint32_t b0 = to_tf32(qv(k0 + tq, cc + gq));
        const uint32_t b1 = to_tf32(qv(k0 + tq + 4, cc + gq));
        mma1688_tf32(acc, a, b0, b1);
    }
    C[(cr + gq) * ldc + cc + 2 * tq] = sign * acc[0];
    C[(cr + gq) * ldc + cc + 2 * tq + 1] = sign * acc[1];
    C[(cr + gq + 8) * ldc + cc + 2 * tq] = sign * acc[2];
    C[(cr + gq + 8) * ldc + cc + 2 * tq + 1] = sign * acc[3];
}

// Barrier of the first n threads of the CTA (id 1-15; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Warps 0-7 join the two inverted 32 x 32 diagonal blocks: one 16 x 8 tile of
// T = A21 X11 per warp, a barrier of the eight warps, one tile of X21 = -X22 T.
// No trailing barrier (the caller's follows).
__device__ __forceinline__ void inv_join64(float* X, const float* A, float* T, int warp, int lane) {
    constexpr int N = 32;
    const int cr = (warp >> 2) * 16, cc = (warp & 3) * 8;
    tile_mm_tf32<N, false, true>(A + N * AP, AP, X, AP, T, N, cr, cc, 1.f, lane);
    named_sync(2, 256);
    tile_mm_tf32<N, true, false>(X + N * AP + N, AP, T, N, X + N * AP, AP, cr, cc, -1.f, lane);
}

// One warp joins the two inverted 16 x 16 diagonal blocks of the 32-block at rows
// 32 p ..: T = A21 X11, then X21 = -X22 T (two 16 x 8 tiles per product, ordered
// by __syncwarp, no CTA barrier).
__device__ __forceinline__ void inv_join16_warp(float* X, const float* A, float* T, int p, int lane) {
    const int r1 = 32 * p, r2 = r1 + 16;
    tile_mm_tf32<16, false, true>(A + r2 * AP + r1, AP, X + r1 * AP + r1, AP, T, 16, 0, 0, 1.f, lane);
    tile_mm_tf32<16, false, true>(A + r2 * AP + r1, AP, X + r1 * AP + r1, AP, T, 16, 0, 8, 1.f, lane);
    __syncwarp();
    tile_mm_tf32<16, true, false>(X + r2 * AP + r2, AP, T, 16, X + r2 * AP + r1, AP, 0, 0, -1.f, lane);
    tile_mm_tf32<16, true, false>(X + r2 * AP + r2, AP, T, 16, X + r2 * AP + r1, AP, 0, 8, -1.f, lane);
}

__device__ __forceinline__ void raise_timeout(uint8_t* ws, volatile int* abort) {
    *abort = 1;
    atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
}

// Issues the level-pair product D[tmem] = Aop Bop^T (M = 128, N = 64, K = DK, both
// operands M/N-major bf16) from one operand buffer, then commits to `bar`.
template <int DK>
__device__ __forceinline__ void issue_level_pair(uint32_t tmem, const uint8_t* buf, uint64_t* bar) {
    constexpr uint32_t id = ptx::idesc_bf16(128, 64) | kAMajorMN | kBMajorMN;
    constexpr uint32_t sbo = (DK / 8) * 128;
    const uint32_t a = ptx::smem_u32(buf), b = a + 128 * DK * 2;
    const uint64_t ad = ptx::smem_desc(a, 128, sbo), bd = ptx::smem_desc(b, 128, sbo);
#pragma unroll
    for (int kk = 0; kk < DK / 16; ++kk)  // K = 16 per step: two 128-byte core columns
        ptx::mma_bf16(tmem, ad + (uint64_t)((kk * 256) >> 4), bd + (uint64_t)((kk * 256) >> 4), id,
                      kk > 0);
    ptx::mma_commit(bar);
}

// tmq .. tmg: addresses of __grid_constant__ kernel parameters.  smem_raw: the
// kernel's dynamic shared memory (1024-byte aligned, sizeof(FactorSmem) bytes).
// plan.ut: u leaves as [64/4][dv][4] fp32 (a float4 of 4 consecutive rows per value
// column, columns fastest: a warp of consecutive columns reads 4 rows of each with
// one contiguous 512-byte load) instead of the slabbed U0 layout; with bf16 inputs
// and dv = 128 the product itself is transposed (u^T, M = dv), so that every
// thread leaves with four 16-byte stores.  (A runtime choice, uniform over the CTA:
// one copy of the body serves both layouts.)
template <int DK, int DV, typename TIn, typename TG>
__device__ __forceinline__ void factor_body(const Dims& d, const CUtensorMap* tmq, const CUtensorMap* tmk,
                                            const CUtensorMap* tmv, const CUtensorMap* tmg,
                                            const float* __restrict__ beta, uint8_t* __restrict__ ws,
                                            uint8_t* smem_raw, const ItemPlan plan) {
    const CUtensorMap &tm_q = *tmq, &tm_k = *tmk, &tm_v = *tmv, &tm_g = *tmg;
    using Sm = FactorSmem<DK, DV, TIn>;
    using Cf = FactorCfg<DK, DV, TIn>;
    constexpr bool kBf16In = sizeof(TIn) == 2;
    // u^T straight from the tensor cores (bf16 inputs, dv = 128: the M = dv product)
    const bool UT = plan.ut;
    const bool kUTmma = UT && kBf16In && DV == 128;
    constexpr int CPT = DK / 64;  // channels per thread in the level phase
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    const WsLayout W(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    const int4* chunk_tab = reinterpret_cast<const int4*>(ws + W.chunks);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = d.H;
    const FactorLayout F(DK, DV);
    volatile int* abort = &sm.abort;

    if (tid == 0) {
        ptx::mbar_init(&sm.ld_bar, 1);
        ptx::mbar_init(&sm.v_bar, 1);
        for (int i = 0; i < 3; ++i) ptx::mbar_init(&sm.lv_bar[i], 1);
        ptx::mbar_init(&sm.wu_bar, 2);  // u and w^T, two issuing threads
        ptx::mbar_init(&sm.drain_bar, 3);
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

    // Persistent: items are (chunk, head) pairs over the schedule's chunks at
    // positions plan.first + n * plan.stride of the plan's order; h == H marks the
    // end.  (With a list, an item's position is known an iteration before its list
    // entry is needed, so the load is issued early.)
    const int total = hdr->total_chunks;
    const int n_items = total * H;
    struct Item { int c, h, i; };
    auto item_at = [&](int i) -> Item {
        if (i >= n_items) return Item{0, H, i};
        if (plan.list) {
            const int v = plan.list[i];
            return Item{v / H, v % H, i};
        }
        return Item{i % total, i / total, i};
    };
    auto advance = [&](Item a) { return item_at(a.i + plan.stride); };
    auto rows_of = [&](Item it) {  // {first token row, valid rows} (zeros past the last item)
        if (it.h >= H) return make_int2(0, 0);
        const int4 t = chunk_tab[it.c];
        return make_int2(t.y, t.z);
    };

    // Tensor copies (one thread).  q, k, g complete on ld_bar; v on v_bar (bf16
    // inputs: it is needed only by the last products, so it may arrive late), or
    // with the others on ld_bar into the ring (fp32 inputs, converted in P1).
    constexpr uint32_t QB = DK * sizeof(TIn), GB = DK * sizeof(TG), VB = DV * sizeof(TIn);
    uint8_t* const st_g = reinterpret_cast<uint8_t*>(sm.gr);
    // phases of ld_bar / v_bar issued and seen complete (thread 0), so that copies
    // still in flight when the CTA leaves early can be waited for
    uint32_t ld_issued = 0, ld_done = 0, v_issued = 0, v_done = 0;
    auto issue_qkg = [&](Item it, int2 nk) {
        ptx::mbar_arrive_expect_tx(&sm.ld_bar, (uint32_t)kChunk * (2 * QB + GB + (kBf16In ? 0 : VB)));
        ptx::tma_load_3d(sm.qr, &tm_q, 0, it.h, nk.x, &sm.ld_bar);
        ptx::tma_load_3d(sm.kr, &tm_k, 0, it.h, nk.x, &sm.ld_bar);
        ptx::tma_load_3d(st_g, &tm_g, 0, it.h, nk.x, &sm.ld_bar);
        if (!kBf16In) ptx::tma_load_3d(sm.ring, &tm_v, 0, it.h, nk.x, &sm.ld_bar);
        ++ld_issued;
    };
    auto issue_v = [&](Item it, int2 nk) {  // bf16 inputs only
        ptx::mbar_arrive_expect_tx(&sm.v_bar, (uint32_t)kChunk * DV * 2);
        ptx::tma_load_4d(sm.vs, &tm_v, 0, nk.x, it.h, 0, &sm.v_bar);
        ++v_issued;
    };
    // beta of row t of an item, for the thread that will be thread t of that item's P1
    float rb = 0.f;
    auto load_beta = [&](Item it, int2 nk, int t) {
        rb = (t >= 0 && t < kChunk && t < nk.y) ? beta[(size_t)(nk.x + t) * H + it.h] : 0.f;
    };

    Item item = item_at(plan.first);
    int2 rows_cur = rows_of(item);
    Item next = advance(item), after = advance(next);  // carried from item to item
    int2 rows_next = rows_of(next), rows_after = rows_of(after);
    if (item.h < H) {
        if (tid == 0) {
            issue_qkg(item, rows_cur);
            if (kBf16In) issue_v(item, rows_cur);
        }
        load_beta(item, rows_cur, tid);
    }
    uint32_t par = 0;  // every per-item barrier completes once per item
    // Tensor memory: item n works in columns [256 (n % 2), + 192) (level products,
    // then u and w^T), so that its u and w^T can wait there while item n + 1 runs;
    // they leave during item n + 1's last products (or after the last item).
    auto epilogue = [&](uint32_t reg, uint8_t* wq_dst, float* u_dst) {
        const int q = warp & 3, cg = warp >> 2;
        // w^T: lane = channel (dk = 64: lanes 0-15 of each quarter), columns = chunk rows
        {
            float x[16];
            ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + reg + 16 * cg, x);
            ptx::tmem_ld_wait();
            const int cc = DK == 128 ? 32 * q + lane : 16 * q + lane;
            if (DK == 128 || lane < 16) {
                float y0[8], y1[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    y0[u] = x[u];
                    y1[u] = x[8 + u];
                }
                *reinterpret_cast<uint4*>(wq_dst + mn_off<DK>(16 * cg, cc)) = pack8(y0);
                *reinterpret_cast<uint4*>(wq_dst + mn_off<DK>(16 * cg + 8, cc)) = pack8(y1);
            }
        }
        if (kUTmma) {
            // u^T: lane = value column 32 q + lane, columns = chunk rows 16 cg ..: four
            // float4 of 4 rows each, a warp's 32 columns contiguous ([64/4][dv][4])
            float x[16];
            ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + reg + 64 + 16 * cg, x);
            ptx::tmem_ld_wait();
            float4* const dst = reinterpret_cast<float4*>(u_dst) + 4 * cg * DV + 32 * q + lane;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
                dst[k4 * DV] = make_float4(x[4 * k4], x[4 * k4 + 1], x[4 * k4 + 2], x[4 * k4 + 3]);
            return;
        }
        // u: lanes 0-15 of each quarter = chunk rows 16 q .., columns DV/4 per warp
        {
            constexpr int NC = DV / 4;
            const int row = 16 * q + lane;
#pragma unroll
            for (int i = 0; i < NC / 16; ++i) {
                float x[16];
                ptx::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + reg + 64 + cg * NC + 16 * i, x);
                ptx::tmem_ld_wait();
                if (lane < 16) {
                    if (UT) {  // [64/4][dv][4]: a float4 of 4 consecutive rows per column
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            u_dst[((row >> 2) * DV + cg * NC + 16 * i + e) * 4 + (row & 3)] = x[e];
                    } else {
#pragma unroll
                        for (int u4 = 0; u4 < 4; ++u4) {
                            const int n = cg * NC + 16 * i + 4 * u4;
                            *reinterpret_cast<float4*>(&u_dst[u0_index(row, n)]) =
                                make_float4(x[4 * u4], x[4 * u4 + 1], x[4 * u4 + 2], x[4 * u4 + 3]);
                        }
                    }
                }
            }
        }
    };
    // ------------------------------------------------------------ P1: load
    // Row norms of q and k, and beta, of the item with L valid rows whose copies
    // complete phase pp of ld_bar, by threads t = 0 .. NT-1 of the CTA (all of them,
    // or warps 8-15 while warps 0-7 invert the previous item's matrix); no barrier
    // inside.  Rows past the chunk end get zero norms (so qh = kh = 0 there) and beta
    // = 0.  beta of this thread's row arrived in rb (load_beta).
    auto p1 = [&](const int L, const uint32_t pp, const int t, auto nt_c, float* bsdst) {
        {
            if (ptx::mbar_wait_or_abort(&sm.ld_bar, pp, abort)) {
                if (tid == 0) ++ld_done;
            } else {
                raise_timeout(ws, abort);
            }
            constexpr int NT = decltype(nt_c)::value;  // threads taking part
            // CH channels a thread (16, or 8 when every thread is needed for a row),
            // CPR threads a row, NP rows a thread; all loads first, then the NP
            // independent reductions side by side
            constexpr int CPR = DK / 16 > NT / kChunk ? DK / 16 : NT / kChunk;
            constexpr int CH = DK / CPR, RP = NT / CPR, NP = kChunk / RP;
            static_assert(CH % 8 == 0 && NP >= 1, "row split");
            constexpr int QW = CH * (int)sizeof(TIn) / 16;  // 16-byte words a thread reads
            static_assert(QW * CPR * 16 == (int)QB, "a row is read once");
            const int ck = t % CPR, rsub = t / CPR;
            float sq[NP], sk[NP];
    #pragma unroll
            for (int p = 0; p < NP; ++p) {
                const int r = rsub + p * RP;
                // word ck + w2 * CPR of the row: each load of a warp is contiguous
                const uint4* wq = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(sm.qr) + r * QB) + ck;
                const uint4* wk = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(sm.kr) + r * QB) + ck;
                uint4 rq[QW], rk[QW];
    #pragma unroll
                for (int w2 = 0; w2 < QW; ++w2) {
                    rq[w2] = wq[w2 * CPR];
                    rk[w2] = wk[w2 * CPR];
                }
                sq[p] = 0.f;
                sk[p] = 0.f;
    #pragma unroll
                for (int h8 = 0; h8 < CH / 8; ++h8) {
                    float xq[8], xk[8];
                    unpack8<TIn>(rq + h8 * (QW * 8 / CH), xq);
                    unpack8<TIn>(rk + h8 * (QW * 8 / CH), xk);
    #pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sq[p] = fmaf(xq[e], xq[e], sq[p]);
                        sk[p] = fmaf(xk[e], xk[e], sk[p]);
                    }
                }
            }
    #pragma unroll
            for (int o = 1; o < CPR; o <<= 1) {
    #pragma unroll
                for (int p = 0; p < NP; ++p) {
                    sq[p] += __shfl_xor_sync(0xffffffffu, sq[p], o);
                    sk[p] += __shfl_xor_sync(0xffffffffu, sk[p], o);
                }
            }
            if (ck == 0) {
    #pragma unroll
                for (int p = 0; p < NP; ++p) {
                    const int r = rsub + p * RP;
                    sm.iq[r] = r < L ? rsqrtf(sq[p] + 1e-6f) : 0.f;
                    sm.ik[r] = r < L ? rsqrtf(sk[p] + 1e-6f) : 0.f;
                }
            }
            if constexpr (!kBf16In) {  // fp32 v (in the ring) -> the tf32 K-major operand, zero past the end
                const float* vr = reinterpret_cast<const float*>(sm.ring);
                for (int e = t; e < (kChunk / 4) * DV; e += NT) {
                    const int n = e % DV, r4 = 4 * (e / DV);  // a warp: 32 consecutive columns
                    float4 x4;
                    x4.x = r4 < L ? vr[r4 * DV + n] : 0.f;
                    x4.y = r4 + 1 < L ? vr[(r4 + 1) * DV + n] : 0.f;
                    x4.z = r4 + 2 < L ? vr[(r4 + 2) * DV + n] : 0.f;
                    x4.w = r4 + 3 < L ? vr[(r4 + 3) * DV + n] : 0.f;
                    *reinterpret_cast<float4*>(&sm.vs[op_index32(n, r4, DV)]) = x4;
                }
            }
            if (t < kChunk) bsdst[t] = rb;
        }
    };
    // Warm L2 with an item's inputs, so that its tensor copies find them there.
    auto warm_l2 = [&](Item y, int2 ry) {
        if (y.h < H) {
            ptx::tma_prefetch_3d(&tm_q, 0, y.h, ry.x);
            ptx::tma_prefetch_3d(&tm_k, 0, y.h, ry.x);
            ptx::tma_prefetch_3d(&tm_g, 0, y.h, ry.x);
            if (kBf16In) ptx::tma_prefetch_4d(&tm_v, 0, ry.x, y.h, 0);
            else ptx::tma_prefetch_3d(&tm_v, 0, y.h, ry.x);
        }
    };
    using AllThreads = std::integral_constant<int, kThreads>;
    using HalfThreads = std::integral_constant<int, kThreads / 2>;
    // bf16 inputs: the next item's P1 runs on warps 8-15 while warps 0-7 invert this
    // item's matrix; fp32 inputs: at the start of each item (its v tile lands in the
    // ring, which the inversion uses)
    bool p1_done = false;

    bool have_prev = false;
    uint32_t prev_reg = 0;
    Item prev_item{0, H, 0};
    bool pub_pending = false;  // with ready flags: an item complete but not yet published
    Item pub_item{0, H, 0};
    uint8_t* prev_wq = nullptr;
    float* prev_u = nullptr;
    while (item.h < H) {
    const uint32_t reg = par ? 256u : 0u;
    const int c = item.c, h = item.h;
    const Item y = advance(after);  // the item after `after` (its rows: before P5)
    uint8_t* const fb = ws + W.factors + ((size_t)c * H + h) * W.factor_bytes;
    uint8_t* const gWQ = fb + F.wq;  // [w; QG], M-major, 128 x DK bf16
    float* const gKT = reinterpret_cast<float*>(fb + F.kt);
    __nv_bfloat16* const gP = reinterpret_cast<__nv_bfloat16*>(fb + F.p);
    float* const gU = reinterpret_cast<float*>(fb + F.u0);
    float* const gGL = reinterpret_cast<float*>(fb + F.gl);
    const int L = rows_cur.y;

    if (!p1_done) {
        p1(L, par, tid, AllThreads{}, sm.bs[par]);
        __syncthreads();
        if (tid == 64) warm_l2(after, rows_after);
    }
    p1_done = false;
    // rb: beta of the next item, for its P1 (run by warps 8-15 with bf16 inputs)
    if (next.h < H) load_beta(next, rows_next, kBf16In ? tid - kThreads / 2 : tid);

    // ------------------------------------------ P2: level operands, QG, KT, kh gamma
    // Thread: 8-row block b = warp / 2 (rows 8b .. 8b+7) of CPT channels
    // c_j = (warp % 2) * DK/2 + lane + 32 j; lanes hold consecutive channels, so every
    // 16-byte operand row a warp writes is contiguous with its neighbours'.
    {
        const int b = warp >> 1, hf = warp & 1;
        float a[CPT][8], kh[CPT][8], qh[CPT][8];
        float dg[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) dg[u] = 0.f;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int cc = hf * (DK / 2) + lane + 32 * j;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int r = 8 * b + u;
                a[j][u] = r < L ? __expf(to_f(reinterpret_cast<const TG*>(sm.gr)[r * DK + cc])) : 1.f;
                kh[j][u] = to_f(sm.kr[r * DK + cc]) * sm.ik[r];
                qh[j][u] = to_f(sm.qr[r * DK + cc]) * sm.iq[r];
                dg[u] = fmaf(qh[j][u], kh[j][u], dg[u]);
            }
            float t8 = a[j][1];
#pragma unroll
            for (int u = 2; u < 8; ++u) t8 *= a[j][u];
            sm.blk_a[b * DK + cc] = a[j][0];
            sm.blk_t[b * DK + cc] = t8;
        }
        // level pair 0: s = 1 (rows [kh R; qh R] at ranks 0-63, columns at 0-31) and
        // s = 2 (ranks 64-127, columns 32-63); all factors are local to the block
        uint8_t* const p0 = sm.ring;
        uint8_t* const p0b = sm.ring + 128 * DK * 2;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int cc = hf * (DK / 2) + lane + 32 * j;
            const float* x = a[j];
            const float* k = kh[j];
            const float* q = qh[j];
            const int m = 4 * b;
            // s = 1: rows 1, 3, 5, 7 (factor 1); columns 0, 2, 4, 6 (factor alpha of the next row)
            st4<DK>(p0, m, cc, k[1], k[3], k[5], k[7]);
            st4<DK>(p0, 32 + m, cc, q[1], q[3], q[5], q[7]);
            st4<DK>(p0b, m, cc, k[0] * x[1], k[2] * x[3], k[4] * x[5], k[6] * x[7]);
            // s = 2: rows 2, 3, 6, 7 (factors 1, a3, 1, a7); columns 0, 1, 4, 5 (to rows 2 / 6)
            st4<DK>(p0, 64 + m, cc, k[2], k[3] * x[3], k[6], k[7] * x[7]);
            st4<DK>(p0, 96 + m, cc, q[2], q[3] * x[3], q[6], q[7] * x[7]);
            st4<DK>(p0b, 32 + m, cc, k[0] * (x[1] * x[2]), k[1] * x[2], k[4] * (x[5] * x[6]), k[5] * x[6]);
        }
        // qh . kh of the 8 rows: reduce over the warp's 32 channels (halving, 9
        // shuffles); lane l ends with row (l >> 2) & 7
        {
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float h4[4], h2[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float send = b4 ? dg[i] : dg[i + 4];
                h4[i] = (b4 ? dg[i + 4] : dg[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float send = b3 ? h4[i] : h4[i + 2];
                h2[i] = (b3 ? h4[i + 2] : h4[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            const float send = b2 ? h2[0] : h2[1];
            float h1 = (b2 ? h2[1] : h2[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
            h1 += __shfl_xor_sync(0xffffffffu, h1, 2);
            h1 += __shfl_xor_sync(0xffffffffu, h1, 1);
            if ((lane & 3) == 0) sm.diag[hf * kChunk + 8 * b + ((lane >> 2) & 7)] = h1;
        }
        ptx::fence_proxy_async_smem();  // operand writes (and the input reads) before async-proxy use
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (tid == 0 && !*abort) {
            issue_level_pair<DK>(tmem + reg + 0, sm.ring, &sm.lv_bar[0]);
            // q, k and g of this item are in registers now: the next item's copies may land
            if (kBf16In && next.h < H) issue_qkg(next, rows_next);
        }

        // per-channel block scalars: ba = alpha at a block's first row, bt = alpha
        // over its rows 1..7, e = ba bt = alpha over the whole block (register
        // copies are indexed by constants only; the block's neighbours' values that
        // depend on this warp's block come straight from shared memory)
        auto load_blk = [&](int cc, float (&ba)[8], float (&bt)[8]) {
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                ba[bb] = sm.blk_a[bb * DK + cc];
                bt[bb] = sm.blk_t[bb * DK + cc];
            }
        };
        // level pair 1: s = 4 (local) and s = 8 (odd blocks: prefix from the block
        // start; even blocks: suffix up to the next block's first row)
        uint8_t* const p1 = Cf::NBUF == 2 ? sm.ring + Cf::PAIR : sm.ring;
        if (Cf::NBUF == 1) {
            if (!ptx::mbar_wait_or_abort(&sm.lv_bar[0], par, abort)) raise_timeout(ws, abort);
        }
        uint8_t* const p1b = p1 + 128 * DK * 2;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int cc = hf * (DK / 2) + lane + 32 * j;
            const float* x = a[j];
            const float* k = kh[j];
            const float* q = qh[j];
            float ba[8], bt[8];
            load_blk(cc, ba, bt);
            const int m = 4 * b;
            // s = 4: rows 4-7 (factors 1, a5, a5a6, a5a6a7), columns 0-3 (suffixes to row 4)
            const float r5 = x[5], r6 = r5 * x[6], r7 = r6 * x[7];
            st4<DK>(p1, m, cc, k[4], k[5] * r5, k[6] * r6, k[7] * r7);
            st4<DK>(p1, 32 + m, cc, q[4], q[5] * r5, q[6] * r6, q[7] * r7);
            const float c3 = x[4], c2 = x[3] * c3, c1 = x[2] * c2, c0 = x[1] * c1;
            st4<DK>(p1b, m, cc, k[0] * c0, k[1] * c1, k[2] * c2, k[3] * c3);
            // s = 8
            float pre[8], suf[8];
            pre[0] = 1.f;
#pragma unroll
            for (int u = 1; u < 8; ++u) pre[u] = pre[u - 1] * x[u];
            suf[7] = 1.f;
#pragma unroll
            for (int u = 6; u >= 0; --u) suf[u] = suf[u + 1] * x[u + 1];
            const int m8 = (b >> 1) * 8;
            if (b & 1) {
                float vk[8], vq[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    vk[u] = k[u] * pre[u];
                    vq[u] = q[u] * pre[u];
                }
                st8<DK>(p1, 64 + m8, cc, vk);
                st8<DK>(p1, 96 + m8, cc, vq);
            } else {
                const float an = sm.blk_a[(b + 1) * DK + cc];
                float vc[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) vc[u] = k[u] * (suf[u] * an);
                st8<DK>(p1b, 32 + m8, cc, vc);
            }
            // whole-chunk factors: gamma_r = (alpha over rows 0..r), gamma_L / gamma_r
            // = (alpha over rows r+1..63)
            float gin = 1.f, sout = 1.f;
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                const float e = ba[bb] * bt[bb];
                if (bb < b) gin *= e;
                if (bb > b) sout *= e;
            }
            const float g0 = gin * x[0];
            float vg[8], vk[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float gam = g0 * pre[u];
                vg[u] = q[u] * gam;
                vk[u] = k[u] * gam;
            }
            // QG: rows 64 + 8b .. of the [w; QG] tile (global, M-major)
            *reinterpret_cast<uint4*>(gWQ + mn_off<DK>(kChunk + 8 * b, cc)) = pack8(vg);
            // (kh gamma)^T for the w product: K-major operand, 8 chunk rows of channel cc
            // (fp32 inputs: tf32, in the q staging, whose reads all came before the
            // barrier above)
            if constexpr (kBf16In) {
                *reinterpret_cast<uint4*>(&sm.kg[op_index(cc, 8 * b, DK)]) = pack8(vk);
            } else {
                float* kgf = reinterpret_cast<float*>(sm.qr);
                *reinterpret_cast<float4*>(&kgf[op_index32(cc, 8 * b, DK)]) = make_float4(vk[0], vk[1], vk[2], vk[3]);
                *reinterpret_cast<float4*>(&kgf[op_index32(cc, 8 * b + 4, DK)]) = make_float4(vk[4], vk[5], vk[6], vk[7]);
            }
            // KT (fp32, tf32 operand layout): kh * gamma_L / gamma
            float kt[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) kt[u] = k[u] * (suf[u] * sout);
            *reinterpret_cast<float4*>(&gKT[op_index32(cc, 8 * b, DK)]) = make_float4(kt[0], kt[1], kt[2], kt[3]);
            *reinterpret_cast<float4*>(&gKT[op_index32(cc, 8 * b + 4, DK)]) = make_float4(kt[4], kt[5], kt[6], kt[7]);
            if (b == 7) gGL[cc] = g0 * pre[7];
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if (tid == 0 && !*abort) issue_level_pair<DK>(tmem + reg + 64, p1, &sm.lv_bar[1]);

        // level pair 2: s = 16 and s = 32, into the buffer of pair 0 once its
        // product has completed (with one buffer: once pair 1's has)
        if (!ptx::mbar_wait_or_abort(&sm.lv_bar[Cf::NBUF == 2 ? 0 : 1], par, abort)) raise_timeout(ws, abort);
        uint8_t* const p2 = sm.ring;
        uint8_t* const p2b = sm.ring + 128 * DK * 2;
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int cc = hf * (DK / 2) + lane + 32 * j;
            const float* x = a[j];
            const float* k = kh[j];
            const float* q = qh[j];
            float pre[8], suf[8];
            pre[0] = 1.f;
#pragma unroll
            for (int u = 1; u < 8; ++u) pre[u] = pre[u - 1] * x[u];
            suf[7] = 1.f;
#pragma unroll
            for (int u = 6; u >= 0; --u) suf[u] = suf[u + 1] * x[u + 1];
            float ba[8], bt[8], e[8];
            load_blk(cc, ba, bt);
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) e[bb] = ba[bb] * bt[bb];
            // s = 16: blocks 4p, 4p+1 are the lower half (columns), 4p+2, 4p+3 the upper
            {
                const int bq = b & 3;
                const int m16 = (b >> 2) * 16 + (b & 1) * 8;
                if (bq >= 2) {
                    const float cr = bq == 2 ? 1.f : sm.blk_t[(b - 1) * DK + cc] * sm.blk_a[b * DK + cc];
                    float vk[8], vq[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        vk[u] = k[u] * (cr * pre[u]);
                        vq[u] = q[u] * (cr * pre[u]);
                    }
                    st8<DK>(p2, m16, cc, vk);
                    st8<DK>(p2, 32 + m16, cc, vq);
                } else {
                    const float cl = bq == 1 ? sm.blk_a[(b + 1) * DK + cc]
                                            : sm.blk_a[(b + 1) * DK + cc] * sm.blk_t[(b + 1) * DK + cc] *
                                                  sm.blk_a[(b + 2) * DK + cc];
                    float vc[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) vc[u] = k[u] * (suf[u] * cl);
                    st8<DK>(p2b, m16, cc, vc);
                }
            }
            // s = 32: blocks 0-3 are the lower half, 4-7 the upper
            {
                const int m32 = (b & 3) * 8;
                if (b >= 4) {
                    float cr = 1.f;
                    if (b > 4) {
                        cr = bt[4];
#pragma unroll
                        for (int bb = 5; bb < 8; ++bb)
                            if (bb < b) cr *= e[bb];
                        cr *= sm.blk_a[b * DK + cc];
                    }
                    float vk[8], vq[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        vk[u] = k[u] * (cr * pre[u]);
                        vq[u] = q[u] * (cr * pre[u]);
                    }
                    st8<DK>(p2, 64 + m32, cc, vk);
                    st8<DK>(p2, 96 + m32, cc, vq);
                } else {
                    float cl = ba[4];
#pragma unroll
                    for (int bb = 1; bb < 4; ++bb)
                        if (bb > b) cl *= e[bb];
                    float vc[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) vc[u] = k[u] * (suf[u] * cl);
                    st8<DK>(p2b, 32 + m32, cc, vc);
                }
            }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        // (warp 12 has no part in P3, so its issue time hides there)
        if (tid == kIssuer3 && !*abort) issue_level_pair<DK>(tmem + reg + 128, p2, &sm.lv_bar[2]);
    }

    // ------------------------------------------ P3: A and P out of tensor memory
    // Warps 0-11: pair p = warp / 4 and lane quarter q = warp % 4: rows kh R (A) of
    // level 2p + q/2 for even q, qh R (P) for odd q; 32 columns per level.  Lane r
    // holds row i of its level; its columns n in the same 2s-block are j = n + blk s.
    // A and P land row-major in fp32 (row stride 65: the lanes' rows hit distinct
    // banks).
    {
        bool ok = ptx::mbar_wait_or_abort(&sm.lv_bar[1], par, abort);
        ok = ptx::mbar_wait_or_abort(&sm.lv_bar[2], par, abort) && ok;
        if (!ok) raise_timeout(ws, abort);
        ptx::tc_fence_after();
        float* const A = reinterpret_cast<float*>(sm.ring + kOffA);
        float* const Pst = reinterpret_cast<float*>(sm.ring + kOffPst);
        if (warp < 12) {
            const int p = warp >> 2, q = warp & 3;
            const int lg = 2 * p + (q >> 1), s = 1 << lg;
            float v0[16], v1[16];
            const uint32_t col = tmem + ((uint32_t)(32 * q) << 16) + reg + 64 * p + 32 * (q >> 1);
            ptx::tmem_ld16(col, v0);
            ptx::tmem_ld16(col + 16, v1);
            ptx::tmem_ld_wait();
            auto v = [&](int n) { return n < 16 ? v0[n] : v1[n - 16]; };
            const int blk = lane >> lg;                      // the 2s-block of this row
            const int i = (blk << (lg + 1)) + s + (lane & (s - 1));
            float* const row = ((q & 1) == 0 ? A : Pst) + i * AP + (blk << lg);  // + n = column j
            const float sc = (q & 1) == 0 ? sm.bs[par][i] : 1.f;
#pragma unroll
            for (int n = 0; n < 32; ++n)
                if ((n >> lg) == blk) row[n] = sc * v(n);
        }
    }
    const int2 rows_y = rows_of(y);
    ptx::tc_fence_before();
    __syncthreads();
    // ------------------------------------- P5: X = (I + A)^-1 by recursive doubling
    // The four 16 x 16 diagonal blocks by forward substitution in fp32 registers
    // (warp w, lanes 0-15: the columns of block w; right-looking, so each step's
    // dependent chain is one FMA; written whole, zeros above the diagonal).  Then
    // X21 = -X22 (A21 X11) joins two inverted blocks into one twice as large: 16 -> 32
    // by one warp per 32-block on its own, 32 -> 64 by eight warps (mma.sync on tf32
    // inputs, fp32 accumulation).  The upper-right block of each joined 32-block is
    // never written; the 64-join reads it as zero.  Only entries of A strictly below
    // the diagonal are read.
    {
        float* const A = reinterpret_cast<float*>(sm.ring + kOffA);
        float* const X = reinterpret_cast<float*>(sm.ring + kOffX);
        float* const T = reinterpret_cast<float*>(sm.ring + kOffScr);
        if (warp < 8) {
            if (warp < 4) {
                if (lane < 16) {
                    const int base = 16 * warp, jc = lane;
                    float x[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) x[i] = (i == jc) ? 1.f : 0.f;
#pragma unroll
                    for (int m = 0; m < 15; ++m) {  // x[m] is final: remove its share from the rows below
                        const float xm = x[m];
#pragma unroll
                        for (int i = m + 1; i < 16; ++i) x[i] = fmaf(-A[(base + i) * AP + base + m], xm, x[i]);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) X[(base + i) * AP + base + jc] = x[i];
                }
                named_sync(3, 128);  // warps 0-3: the four 16-blocks
                if (warp < 2) inv_join16_warp(X, A, T + 256 * warp, warp, lane);
            }
            named_sync(2, 256);      // warps 0-7: the two 32-blocks
            inv_join64(X, A, T, warp, lane);
        } else {
            if (kBf16In && next.h < H) {
                p1(rows_next.y, par ^ 1u, tid - kThreads / 2, HalfThreads{}, sm.bs[par ^ 1u]);
                if (tid == kThreads / 2 + 64) warm_l2(y, rows_y);
            }
            // the item whose last parts left before the previous item's end barrier:
            // published here, where warps 8-15 have slack and its stores have drained
            if (tid == kThreads / 2 && pub_pending) ptx::flag_publish(plan.ready + (size_t)pub_item.c * H + pub_item.h);
        }
        __syncthreads();
        if (kBf16In && next.h < H) {
            p1_done = true;
            if (tid == 0 && !*abort) ++ld_done;  // warps 8-15 saw the next item's copies land
        }
    }

    // ------------------------------------- P6: X Diag(beta) as hi + lo operands
    // (bf16 with bf16 inputs; tf32 with fp32 inputs, whose u and w run on tf32:
    // the hi part in the ring, the lo part in the k staging, dead by then)
    {
        const float* X = reinterpret_cast<const float*>(sm.ring + kOffX);
        // 64 rows x 8 groups: a warp takes 32 consecutive rows of one group, so its
        // X reads (row stride 65) and operand stores (rows of a group are adjacent
        // 16-byte core rows) are free of bank conflicts
        const int i = tid & 63, jb = (tid >> 6) * 8;
        float x[8], lo[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = jb + u;
            x[u] = (j <= i) ? X[i * AP + j] * sm.bs[par][j] : 0.f;
        }
        if constexpr (kBf16In) {
            __nv_bfloat16* xop = reinterpret_cast<__nv_bfloat16*>(sm.ring + kOffXop);
            __nv_bfloat16* xlo = reinterpret_cast<__nv_bfloat16*>(sm.ring + kOffXlo);
            const uint4 hi = pack8(x);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hi);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                lo[2 * u] = x[2 * u] - f.x;
                lo[2 * u + 1] = x[2 * u + 1] - f.y;
            }
            *reinterpret_cast<uint4*>(&xop[op_index(i, jb, kChunk)]) = hi;
            *reinterpret_cast<uint4*>(&xlo[op_index(i, jb, kChunk)]) = pack8(lo);
        } else {
            float* xop = reinterpret_cast<float*>(sm.ring + kOffXop);
            float* xlo = reinterpret_cast<float*>(sm.kr);
            float hi[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                hi[u] = __uint_as_float(to_tf32(x[u]));
                lo[u] = __uint_as_float(to_tf32(x[u] - hi[u]));
            }
#pragma unroll
            for (int h4 = 0; h4 < 8; h4 += 4) {
                *reinterpret_cast<float4*>(&xop[op_index32(i, jb + h4, kChunk)]) =
                    make_float4(hi[h4], hi[h4 + 1], hi[h4 + 2], hi[h4 + 3]);
                *reinterpret_cast<float4*>(&xlo[op_index32(i, jb + h4, kChunk)]) =
                    make_float4(lo[h4], lo[h4 + 1], lo[h4 + 2], lo[h4 + 3]);
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // ------------------------------------------------- P7: u and w^T on tcgen05
    // Two issuing threads (each tcgen05.mma costs its issuer ~85 cycles): thread 0
    // issues u (it needs v) into columns reg + 64 .., thread kIssuer2 issues w^T into
    // columns reg + 0 ..
    if (tid == 0 || tid == kIssuer2) {
        bool okv = true;
        if (kBf16In && tid == 0) {
            okv = ptx::mbar_wait_or_abort(&sm.v_bar, par, abort);
            if (okv) ++v_done;
            else raise_timeout(ws, abort);
        }
        ptx::tc_fence_after();
        if (okv && !*abort && !kBf16In) {  // fp32 inputs: tf32 products, K = 8 per step
            const uint64_t xd[2] = {ptx::smem_desc(ptx::smem_u32(sm.ring + kOffXop), 1024, 128),
                                    ptx::smem_desc(ptx::smem_u32(sm.kr), 1024, 128)};
            if (tid == 0) {  // u = (X Diag(beta)) v, hi then lo
                constexpr uint32_t id_u = ptx::idesc_tf32(kChunk, DV);
                const uint64_t vb = ptx::smem_desc(ptx::smem_u32(sm.vs), (DV / 8) * 128, 128);
                constexpr uint64_t vstep = (uint64_t)((2 * (DV / 8) * 128) >> 4);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 8; ++kk)
                        ptx::mma_tf32(tmem + reg + 64, xd[part] + (uint64_t)(kk * 128), vb + kk * vstep, id_u,
                                      part > 0 || kk > 0);
            } else {         // w^T = (kh gamma)^T (X Diag(beta))^T, hi then lo
                constexpr uint32_t id_w = ptx::idesc_tf32(DK, kChunk);
                const uint64_t kd = ptx::smem_desc(ptx::smem_u32(sm.qr), (DK / 8) * 128, 128);
                constexpr uint64_t kstep = (uint64_t)((2 * (DK / 8) * 128) >> 4);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 8; ++kk)
                        ptx::mma_tf32(tmem + reg + 0, kd + kk * kstep, xd[part] + (uint64_t)(kk * 128), id_w,
                                      part > 0 || kk > 0);
            }
        }
        if (okv && !*abort && kBf16In) {
            const uint64_t xd[2] = {ptx::smem_desc(ptx::smem_u32(sm.ring + kOffXop), 1024, 128),
                                    ptx::smem_desc(ptx::smem_u32(sm.ring + kOffXlo), 1024, 128)};
            if (tid == 0 && kUTmma) {  // u^T = v^T (X Diag(beta))^T (M = dv, v as an M-major A), hi then lo
                constexpr uint32_t id_u = ptx::idesc_bf16(DV, kChunk) | kAMajorMN;
                const uint64_t vb = ptx::smem_desc(ptx::smem_u32(sm.vs), 128, 1024);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk)
                        ptx::mma_bf16(tmem + reg + 64, vb + (uint64_t)(kk * 16), xd[part] + (uint64_t)(kk * 128),
                                      id_u, part > 0 || kk > 0);
            } else if (tid == 0) {  // u = (X Diag(beta)) v, hi then lo
                constexpr uint32_t id_u = ptx::idesc_bf16(kChunk, DV) | kBMajorMN;
                const uint64_t vb = ptx::smem_desc(ptx::smem_u32(sm.vs), 128, 1024);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk)
                        ptx::mma_bf16(tmem + reg + 64, xd[part] + (uint64_t)(kk * 128), vb + (uint64_t)(kk * 16),
                                      id_u, part > 0 || kk > 0);
            } else {         // w^T = (kh gamma)^T (X Diag(beta))^T, hi then lo
                constexpr uint32_t id_w = ptx::idesc_bf16(DK, kChunk);
                const uint64_t kd = ptx::smem_desc(ptx::smem_u32(sm.kg), (DK / 8) * 128, 128);
                constexpr uint64_t kstep = (uint64_t)((2 * (DK / 8) * 128) >> 4);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kChunk / 16; ++kk)
                        ptx::mma_bf16(tmem + reg + 0, kd + kk * kstep, xd[part] + (uint64_t)(kk * 128), id_w,
                                      part > 0 || kk > 0);
            }
        }
        ptx::mma_commit(&sm.wu_bar);  // (also when nothing was issued: the phase still completes)
    }
    // while those products run: P of this item, u and w^T of the previous one
    // P leaves in its operand layout, 16 bytes per thread: row i, columns 8 jb ..;
    // the diagonal (qh_i . kh_i) and the zeros above it are filled in here
    {
        const float* Pst = reinterpret_cast<const float*>(sm.ring + kOffPst);
        const int i = tid >> 3, jb = tid & 7;
        const float dv = sm.diag[i] + sm.diag[kChunk + i];
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = 8 * jb + u;
            x[u] = j < i ? Pst[i * AP + j] : (j == i ? dv : 0.f);
        }
        *reinterpret_cast<uint4*>(&gP[op_index(i, 8 * jb, kChunk)]) = pack8(x);
    }

    // with ready flags, a CTA's first item leaves at once (its consumers start on it)
    const bool first_now = plan.ready != nullptr && !have_prev;
    if (have_prev) epilogue(prev_reg, prev_wq, prev_u);
    if (!ptx::mbar_wait_or_abort(&sm.wu_bar, par, abort)) raise_timeout(ws, abort);
    ptx::tc_fence_after();
    if (first_now) epilogue(reg, gWQ, gU);
    if (tid == 0 && next.h < H && !*abort) {  // v (and, for fp32 inputs, everything) of the next item
        if (kBf16In) issue_v(next, rows_next);
        else issue_qkg(next, rows_next);
    }
    const bool publish_prev = have_prev;  // the previous item's last parts left above
    const Item published = prev_item;
    have_prev = !first_now;
    prev_reg = reg;
    prev_wq = gWQ;
    prev_u = gU;
    prev_item = item;
    ptx::tc_fence_before();
    __syncthreads();
    if (*abort) break;
    pub_pending = plan.ready != nullptr && publish_prev;  // (published during the next item)
    pub_item = published;
    if (first_now && tid == 0) ptx::flag_publish(plan.ready + (size_t)item.c * H + item.h);
    par ^= 1u;
    item = next;
    rows_cur = rows_next;
    next = after;
    rows_next = rows_after;
    after = y;
    rows_after = rows_y;
    }  // items

    if (have_prev) {  // u and w^T of the last item
        ptx::tc_fence_after();
        epilogue(prev_reg, prev_wq, prev_u);
    }

    // Leave cleanly: copies still in flight land, issued MMAs complete, then TMEM goes.
    {
        volatile int never = 0;
        if (tid == 0) {
            for (uint32_t k2 = ld_done; k2 < ld_issued; ++k2) ptx::mbar_wait_or_abort(&sm.ld_bar, k2 & 1u, &never);
            for (uint32_t k2 = v_done; k2 < v_issued; ++k2) ptx::mbar_wait_or_abort(&sm.v_bar, k2 & 1u, &never);
        }
        if (tid == 0 || tid == kIssuer2 || tid == kIssuer3) ptx::mma_commit(&sm.drain_bar);  // each issuer's own products
        if (tid == 0) ptx::mbar_wait_or_abort(&sm.drain_bar, 0, &never);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (plan.ready && tid == 0 && !*abort) {  // the last items' parts all left
        if (pub_pending) ptx::flag_publish(plan.ready + (size_t)pub_item.c * H + pub_item.h);
        if (have_prev) ptx::flag_publish(plan.ready + (size_t)prev_item.c * H + prev_item.h);
    }
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace
}  // namespace kda
