// Per-chunk factors of the chunkwise KDA forward on tensor cores.  Persistent: one
// 512-thread CTA per SM walks (chunk, head) items in steps of the grid size; the
// next item's inputs arrive by TMA tensor copies while the current one finishes,
// and the results leave by bulk copies from shared memory (phases P1-P7 below).
//
// For a chunk of L <= 64 tokens of one sequence and head ("Autoresearch on Kimi
// Delta Attention", section THE MECHANISM: inside a block the work becomes matrix
// products; "NVIDIA Kernel Design Agents optimize Kimi Delta Attention", section 03
// REWARD HACKING: L2 normalisation of q and k, the cumulative decay inside each
// 64-token chunk, the triangular inverse):
//   qh, kh   = rows of q, k over sqrt(|x|^2 + eps)              (fp32)
//   alpha    = exp(g)                                           (one exp per element)
//   A_ij     = beta_i sum_c kh_ic kh_jc D_c(i, j)                 j < i
//   P_ij     = sum_c qh_ic kh_jc D_c(i, j)                        j <= i
//   with D_c(i, j) = exp(Gamma_ic - Gamma_jc) = alpha_c(j+1) ... alpha_c(i)
//   X        = (I + A)^-1                                        (fp32, blocked)
//   [w | u]  = X Diag(beta) [kh * gamma | v]                     (tcgen05, M=64 N=dk+dv K=64,
//                                                                 X Diag(beta) split hi + lo)
//   QG = qh * gamma,  KT = (kh * gamma_L / gamma)^T,  GL = gamma_L,  gamma = exp(Gamma)
// w and QG are written as the two halves of one 128-row operand tile, so that the
// state kernel forms w S and QG S with one M = 128 product.
//
// Every decay factor is a product of alphas over a run of consecutive tokens, so
// it lies in [0, 1]: deep decays underflow to zero and nothing overflows (the
// pages' section 03 describes kernels that formed exp(Gamma) / exp(Gamma') and
// produced NaN).  A and P are split into blocks:
//   * 16 x 16 blocks below the diagonal: with the first row m of the block row as
//     the reference, D(i, j) = D(i, m) D(m, j) factorises into a row factor and a
//     column factor, so the block is a plain product -> mma.sync (bf16, fp32 acc);
//   * the lower-left 8 x 8 quadrant of each diagonal 16-block: the same with the
//     reference at its first row -> mma.sync;
//   * the eight 8 x 8 diagonal blocks: running products per channel (CUDA cores).
#include <cuda.h>          // CUtensorMap (the encoder itself is fetched at run time)
#include <cudaTypedefs.h>  // the encoder's function-pointer type

#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

namespace {

constexpr int kThreads = 512;

template <int DK, int DV, typename TIn>
struct __align__(128) PrepSmem {
    TIn qr[kChunk * DK];   // raw q rows as copied in; qh = qr * iq[row]
    float kn[kChunk * DK]; // kh (fp32), widened in place from the raw rows
    float al[kChunk * DK];
    __nv_bfloat16 vs[kChunk * DV];
    float A[kChunk * (kChunk + 1)];
    float X[kChunk * (kChunk + 1)];
    // mma.sync operands (swizzled bf16 rows of DK), later reused for the tcgen05
    // operands and the inverse's scratch
    union Ops {
        struct {
            __nv_bfloat16 left[48 * DK];    // kh_r D(r, 16R), rows 16..63
            __nv_bfloat16 leftq[48 * DK];   // qh_r D(r, 16R)
            __nv_bfloat16 right[96 * DK];   // kh_j D(16R, j): R=1 rows 0-15, R=2 16-47, R=3 48-95
            __nv_bfloat16 l8[32 * DK];      // kh_r D(r, 16R+8), r in [16R+8, 16R+16)
            __nv_bfloat16 l8q[32 * DK];
            __nv_bfloat16 r8[32 * DK];      // kh_j D(16R+8, j), j in [16R, 16R+8)
        } m;
        struct T {
            __nv_bfloat16 xop[kChunk * kChunk];        // X Diag(beta), operand layout
            __nv_bfloat16 xlo[kChunk * kChunk];        // its rounding remainder (hi + lo split)
            __nv_bfloat16 bop[(DK + DV) * kChunk];     // [kh*gamma | v]^T, operand layout
        } t;
        float scratch[32 * 32];
    } ops;
    float bs[kChunk];
    float iq[kChunk];  // inverse row norms of q (rows past the chunk end are zero)
    float gb[8 * DK];  // alpha(0..8b) per block start b and channel (kept for the w operand)
    float sb[8 * DK];  // alpha(8b+8..63) per block b and channel (kept for KT)
    uint64_t bar;
    uint64_t ld_bar;  // bulk copies of an item's raw inputs
    uint32_t tmem;
    int abort;
};

// 8 elements from 16-byte words: one word of bf16, or two of fp32.
template <typename TIn>
__device__ inline void unpack8(const uint4* w, float (&x)[8]);
template <>
__device__ inline void unpack8<__nv_bfloat16>(const uint4* w, float (&x)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
template <>
__device__ inline void unpack8<float>(const uint4* w, float (&x)[8]) {
    const float* f = reinterpret_cast<const float*>(w);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = f[i];
}

// Two consecutive elements as fp32.
__device__ inline float2 ld2(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ inline float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }

__device__ inline uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ inline uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
}

// Swizzled element offset of (row, k) in a bf16 operand table with DK columns:
// 16-byte chunks XOR-ed with the row's low bits keep mma.sync fragment loads free
// of bank conflicts.
template <int DK>
__device__ inline int sw(int row, int k) {
    return row * DK + ((((k >> 3) ^ (row & 7))) << 3) + (k & 7);
}

template <int DK>
__device__ inline uint32_t lds_pair(const __nv_bfloat16* t, int row, int k) {
    return *reinterpret_cast<const uint32_t*>(t + sw<DK>(row, k));
}

// Packed fp32x2 arithmetic (two lanes of work per instruction).
__device__ inline float2 mul2(float2 a, float2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return *reinterpret_cast<float2*>(&r);
}
__device__ inline float2 scale2(float2 a, float s) { return mul2(a, make_float2(s, s)); }
__device__ inline float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
          "l"(*reinterpret_cast<unsigned long long*>(&c)));
    return *reinterpret_cast<float2*>(&r);
}

__device__ inline void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ inline uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ inline void mma1688_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
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

// Tensor-core join for n = 16, 32: one 16 x 8 tile of T = A21 X11, then of
// X21 = -X22 T, per warp.  Ends with the CTA synchronised.
template <int N>
__device__ __forceinline__ void inv_join_tc(float* X, const float* A, float* T, int warp, int lane) {
    constexpr int AP = kChunk + 1;
    constexpr int PAIRS = kChunk / (2 * N);
    constexpr int TILES = (N / 16) * (N / 8);        // tiles per pair
    for (int t = warp; t < PAIRS * TILES; t += kThreads / 32) {
        const int pidx = t / TILES, tt = t % TILES;
        const int r1 = 2 * pidx * N, r2 = r1 + N;
        const int cr = (tt / (N / 8)) * 16, cc = (tt % (N / 8)) * 8;
        tile_mm_tf32<N, false, true>(A + r2 * AP + r1, AP, X + r1 * AP + r1, AP, T + pidx * N * N,
                                     N, cr, cc, 1.f, lane);
    }
    __syncthreads();
    for (int t = warp; t < PAIRS * TILES; t += kThreads / 32) {
        const int pidx = t / TILES, tt = t % TILES;
        const int r1 = 2 * pidx * N, r2 = r1 + N;
        const int cr = (tt / (N / 8)) * 16, cc = (tt % (N / 8)) * 8;
        tile_mm_tf32<N, true, false>(X + r2 * AP + r2, AP, T + pidx * N * N, N, X + r2 * AP + r1, AP,
                                     cr, cc, -1.f, lane);
    }
    __syncthreads();
}

// Joins pairs of inverted n x n diagonal blocks of X = (I + A)^-1 (row stride
// kChunk + 1): X21 = -X22 (A21 X11).  Upper triangles of X are zero, so the
// products run over full blocks.  Ends with the CTA synchronised.
template <int N>
__device__ __forceinline__ void inv_join(float* X, const float* A, float* T, int tid) {
    constexpr int AP = kChunk + 1;
    constexpr int OUT = (kChunk / (2 * N)) * N * N;
    constexpr int PER = (OUT + kThreads - 1) / kThreads;
#pragma unroll
    for (int qq = 0; qq < PER; ++qq) {
        const int e = tid + qq * kThreads;
        if (e < OUT) {
            const int pidx = e / (N * N), i = (e / N) % N, j = e % N;
            const int r1 = 2 * pidx * N, r2 = r1 + N;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int m = 0; m < N; m += 2) {
                a0 = fmaf(A[(r2 + i) * AP + r1 + m], X[(r1 + m) * AP + r1 + j], a0);
                a1 = fmaf(A[(r2 + i) * AP + r1 + m + 1], X[(r1 + m + 1) * AP + r1 + j], a1);
            }
            T[e] = a0 + a1;
        }
    }
    __syncthreads();
#pragma unroll
    for (int qq = 0; qq < PER; ++qq) {
        const int e = tid + qq * kThreads;
        if (e < OUT) {
            const int pidx = e / (N * N), i = (e / N) % N, j = e % N;
            const int r1 = 2 * pidx * N, r2 = r1 + N;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int m = 0; m < N; m += 2) {
                a0 = fmaf(X[(r2 + i) * AP + r2 + m], T[pidx * N * N + m * N + j], a0);
                a1 = fmaf(X[(r2 + i) * AP + r2 + m + 1], T[pidx * N * N + (m + 1) * N + j], a1);
            }
            X[(r2 + i) * AP + r1 + j] = -(a0 + a1);
        }
    }
    __syncthreads();
}

template <int DK, int DV, typename TIn, typename TG>
__global__ void __launch_bounds__(kThreads, 1)
    prep_tc_kernel(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                   const float* __restrict__ beta, uint8_t* __restrict__ ws) {
    using Sm = PrepSmem<DK, DV, TIn>;
    constexpr int AP = kChunk + 1;
    constexpr int NB = DK + DV;  // columns of the w/u product
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    const WsLayout W(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    const int4* chunk_tab = reinterpret_cast<const int4*>(ws + W.chunks);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = d.H;
    const FactorLayout F(DK, DV);

    if (tid == 0) {
        ptx::mbar_init(&sm.bar, 1);
        ptx::mbar_init(&sm.ld_bar, 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, 256);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    // Persistent: items are (chunk, head) pairs over the schedule's chunks, item
    // i = h * total + c, taken in steps of the grid size (32-bit, no division in the
    // loop: the step is split once into whole heads and a chunk remainder).
    const int total = hdr->total_chunks;
    struct Item { int c, h; };
    const int step_c = total > 0 ? (int)(gridDim.x % (unsigned)total) : 0;
    const int step_h = total > 0 ? (int)(gridDim.x / (unsigned)total) : H;
    auto advance = [&](Item a) {
        a.c += step_c;
        a.h += step_h;
        if (a.c >= total) { a.c -= total; ++a.h; }
        return a;
    };
    // 16-byte load chunks: consecutive lanes take consecutive chunks of a row, so the
    // shared-memory stores are conflict free and a row's lanes reduce its norm.
    constexpr int CPR = DK / 8, RP = kThreads / CPR, NP = kChunk / RP;
    constexpr int VPR = DV / 8, VRP = kThreads / VPR, NVP = kChunk / VRP;
    const int ck = tid % CPR, rsub = tid / CPR;
    const int vk = tid % VPR, vsub = tid / VPR;
    // Raw inputs of an item arrive by tensor copies (TMA: one box of 64 token rows
    // of one head per tensor, rows past the end of the tensor read as zero) into
    // shared regions that are dead while the previous item finishes: q into qr, where
    // it stays (consumers scale it by the row norm), k into kn and g into al (bf16 k
    // and g into the upper halves, widened in place to fp32 once every thread has
    // read its raw words), v into vs (bf16) or, as fp32, into the A and X arrays.
    constexpr bool kBf16In = sizeof(TIn) == 2;
    constexpr bool kBf16G = sizeof(TG) == 2;
    uint8_t* const st_q = reinterpret_cast<uint8_t*>(sm.qr);
    uint8_t* const st_k = reinterpret_cast<uint8_t*>(sm.kn) + (kBf16In ? kChunk * DK * 2 : 0);
    uint8_t* const st_g = reinterpret_cast<uint8_t*>(sm.al) + (kBf16G ? kChunk * DK * 2 : 0);
    uint8_t* const st_v = kBf16In ? reinterpret_cast<uint8_t*>(sm.vs) : reinterpret_cast<uint8_t*>(sm.A);
    static_assert(kBf16In || kChunk * DV * 4 <= 2 * kChunk * (kChunk + 1) * 4, "v staging");
    constexpr uint32_t QB = DK * sizeof(TIn), GB = DK * sizeof(TG), VB = DV * sizeof(TIn);
    // KT staging for its bulk store (two halves of KTH floats).  bf16 inputs: the A
    // array (dead after the inverse) and, at dk = 128, the operand region past the
    // tcgen05 operands -- neither is touched by the next item's copies.  fp32 inputs
    // (their v lands in A): the q array, and the next item's copies are issued only
    // once the store has read it.
    constexpr int KTH = DK * kChunk / 2;
    constexpr size_t kOpsT = sizeof(typename Sm::Ops::T);
    float* const st_kt0 = kBf16In ? sm.A : reinterpret_cast<float*>(sm.qr);
    float* const st_kt1 = (kBf16In && DK == 128)
                              ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(&sm.ops) + kOpsT)
                              : st_kt0 + KTH;
    static_assert(!kBf16In || (DK == 128 ? KTH : 2 * KTH) * 4 <= kChunk * (kChunk + 1) * 4, "KT in A");
    static_assert(!kBf16In || DK != 128 || kOpsT + KTH * 4 <= sizeof(typename Sm::Ops), "KT in ops");
    static_assert(kChunk * DK * 2 + kChunk * DV * 4 <= kOpsT || DK != 128, "w/u staging below KT");
    // Output staging for the bulk stores of w and u (in the operand region).
    __nv_bfloat16* const st_w = reinterpret_cast<__nv_bfloat16*>(&sm.ops);
    float* const st_u = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(&sm.ops) + kChunk * DK * 2);
    static_assert(kChunk * DK * 2 + kChunk * DV * 4 <= sizeof(typename Sm::Ops), "output staging");
    float rb = 0.f;  // beta of this thread's row of the next item (threads < 64)
    // {first token row, valid rows} of an item's chunk (zeros past the last item)
    auto rows_of = [&](Item it) {
        if (it.h >= H) return make_int2(0, 0);
        const int4 t = chunk_tab[it.c];
        return make_int2(t.y, t.z);
    };
    // One thread: the four tensor copies of an item, completing on ld_bar.  Rows
    // of the box past the chunk's end (another sequence's tokens, or zeros past the
    // tensor) are ignored below.
    // With bf16 inputs the q copy goes out early (its array is dead after the diagonal
    // blocks) and the expected bytes of all four are announced with it.
    auto issue_q = [&](Item it, int2 nk) {
        ptx::mbar_arrive_expect_tx(&sm.ld_bar, (uint32_t)kChunk * (2 * QB + GB + VB));
        ptx::tma_load_3d(st_q, &tm_q, 0, it.h, nk.x, &sm.ld_bar);
    };
    auto issue_kgv = [&](Item it, int2 nk) {
        ptx::tma_load_3d(st_k, &tm_k, 0, it.h, nk.x, &sm.ld_bar);
        ptx::tma_load_3d(st_g, &tm_g, 0, it.h, nk.x, &sm.ld_bar);
        ptx::tma_load_3d(st_v, &tm_v, 0, it.h, nk.x, &sm.ld_bar);
    };
    auto issue_copies = [&](Item it, int2 nk) {
        issue_q(it, nk);
        issue_kgv(it, nk);
    };
    auto load_beta = [&](Item it, int2 nk) {
        const int hh = it.h;
        rb = (tid < kChunk && tid < nk.y) ? beta[(size_t)(nk.x + tid) * H + hh] : 0.f;
    };

    Item item = total > 0 ? Item{(int)(blockIdx.x % (unsigned)total), (int)(blockIdx.x / (unsigned)total)}
                          : Item{0, H};
    int2 rows_cur = rows_of(item);
    if (item.h < H) {
        if (tid == 0) issue_copies(item, rows_cur);
        load_beta(item, rows_cur);
    }
    uint32_t ld_phase = 0;
    uint32_t phase = 0;
    while (item.h < H) {
    const int c = item.c, h = item.h;
    const Item next = advance(item), after = advance(next);
    // chunk-table lookups of the next two items, issued now and consumed later
    const int2 rows_next = rows_of(next), rows_after = rows_of(after);
    uint8_t* fb = ws + W.factors + ((size_t)c * H + h) * W.factor_bytes;
    __nv_bfloat16* gWQ = reinterpret_cast<__nv_bfloat16*>(fb + F.wq);  // rows: w, then qh gamma
    float* gKT = reinterpret_cast<float*>(fb + F.kt);
    __nv_bfloat16* gP = reinterpret_cast<__nv_bfloat16*>(fb + F.p);
    float* gU = reinterpret_cast<float*>(fb + F.u0);
    float* gGL = reinterpret_cast<float*>(fb + F.gl);

    // ---------------------------------------------------------------- P1: load
    // (the bulk copies were issued earlier) normalise q and k, alpha = exp(g), stage v
    {
        if (!ptx::mbar_wait_or_abort(&sm.ld_bar, ld_phase, &sm.abort) && tid == 0)
            atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
        ld_phase ^= 1u;
        const int L = rows_cur.y;
        constexpr int QW = (int)sizeof(TIn) / 2;  // 16-byte words per 8 elements
        constexpr int GW = (int)sizeof(TG) / 2;
        uint4 rk[NP][QW], rg[NP][GW];
        float ikr[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int r = rsub + p * RP;
            const bool ok_r = r < L;
            uint4* wq = reinterpret_cast<uint4*>(st_q + r * QB + ck * 8 * sizeof(TIn));
            const uint4* wk = reinterpret_cast<const uint4*>(st_k + r * QB + ck * 8 * sizeof(TIn));
            const uint4* wg = reinterpret_cast<const uint4*>(st_g + r * GB + ck * 8 * sizeof(TG));
            uint4 rq[QW];
#pragma unroll
            for (int w2 = 0; w2 < QW; ++w2) {
                rq[w2] = ok_r ? wq[w2] : make_uint4(0, 0, 0, 0);
                rk[p][w2] = ok_r ? wk[w2] : make_uint4(0, 0, 0, 0);
                if (!ok_r) wq[w2] = make_uint4(0, 0, 0, 0);  // q rows past the chunk: zero
            }
#pragma unroll
            for (int w2 = 0; w2 < GW; ++w2) rg[p][w2] = ok_r ? wg[w2] : make_uint4(0, 0, 0, 0);
            float xq[8], xk[8];
            unpack8<TIn>(rq, xq);
            unpack8<TIn>(rk[p], xk);
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                sq = fmaf(xq[e], xq[e], sq);
                sk = fmaf(xk[e], xk[e], sk);
            }
#pragma unroll
            for (int o = 1; o < CPR; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (ck == 0) sm.iq[r] = rsqrtf(sq + 1e-6f);
            ikr[p] = rsqrtf(sk + 1e-6f);
        }
        // raw bf16 k and g words are read before fp32 rows overwrite them
        if (kBf16In || kBf16G) __syncthreads();
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int r = rsub + p * RP;
            float xk[8], xg[8];
            unpack8<TIn>(rk[p], xk);
            unpack8<TG>(rg[p], xg);
            float* dk_ = &sm.kn[r * DK + ck * 8];
            float* da = &sm.al[r * DK + ck * 8];
#pragma unroll
            for (int e = 0; e < 8; e += 4) {
                *reinterpret_cast<float4*>(dk_ + e) = make_float4(xk[e] * ikr[p], xk[e + 1] * ikr[p],
                                                                  xk[e + 2] * ikr[p], xk[e + 3] * ikr[p]);
                *reinterpret_cast<float4*>(da + e) = make_float4(__expf(xg[e]), __expf(xg[e + 1]),
                                                                 __expf(xg[e + 2]), __expf(xg[e + 3]));
            }
        }
#pragma unroll
        for (int p = 0; p < NVP; ++p) {
            const int r = vsub + p * VRP;
            uint4* dv = reinterpret_cast<uint4*>(&sm.vs[r * DV + vk * 8]);
            if (r >= L) {
                *dv = make_uint4(0, 0, 0, 0);
            } else if (!kBf16In) {  // fp32 v staged in the A / X arrays
                float xv[8];
                unpack8<TIn>(reinterpret_cast<const uint4*>(st_v + r * VB + vk * 8 * sizeof(TIn)), xv);
                *dv = pack8(xv);
            }
        }
        if (tid < kChunk) sm.bs[tid] = rb;
    }
    __syncthreads();

    // Warm L2 with the inputs of the item after next, so that its tensor copies
    // (issued during the next item) find them there.
    if (tid == 64 && after.h < H) {
        const int hy = after.h;
        ptx::tma_prefetch_3d(&tm_q, 0, hy, rows_after.x);
        ptx::tma_prefetch_3d(&tm_k, 0, hy, rows_after.x);
        ptx::tma_prefetch_3d(&tm_g, 0, hy, rows_after.x);
        ptx::tma_prefetch_3d(&tm_v, 0, hy, rows_after.x);
    }

    // ------------------------------------------------ P2: decay products
    if (tid == 0) ptx::bulk_wait_read_all();  // the previous item's stores have left the
                                              // operand region, written again below
    // Every decay factor used below is a product of alpha over a run of rows.  The
    // rows split into eight 8-row blocks; per (block b, channel) the local forward
    // products f_r = alpha(8b+1..r) and backward products g_r = alpha(r+1..8b+7)
    // are formed in registers, and per channel a handful of block scalars join
    // them: Gb_b = alpha(0..8b), Sb_b = alpha(8b+8..63), M(b, R) = alpha(8b+8..16R).
    {
        float* Bi = sm.X;                 // inner block products alpha(8b+1..8b+7) [8][DK]
        float* Gb = sm.gb;                // [8][DK]
        float* Sb = sm.sb;                // [8][DK]
        float* Mt = sm.A;                 // M(b, R): 2 + 4 + 6 rows of [DK]
        constexpr int TPB = kThreads / DK;   // tasks per block pass
        // (a) inner products of every block
        for (int e = tid; e < 8 * DK; e += kThreads) {
            const int bb = e / DK, ch = e % DK;
            float pr = 1.f;
#pragma unroll
            for (int u = 1; u < 8; ++u) pr *= sm.al[(8 * bb + u) * DK + ch];
            Bi[bb * DK + ch] = pr;
        }
        __syncthreads();
        // (b) per-channel block scalars
        if (tid < DK) {
            const int ch = tid;
            float a[8], bi[8];
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                a[bb] = sm.al[(8 * bb) * DK + ch];
                bi[bb] = Bi[bb * DK + ch];
            }
            float gp = a[0];
#pragma unroll
            for (int bb = 0; bb < 8; ++bb) {
                if (bb > 0) gp *= bi[bb - 1] * a[bb];
                Gb[bb * DK + ch] = gp;
            }
            gGL[ch] = gp * bi[7];
            float sp = 1.f;
#pragma unroll
            for (int bb = 7; bb >= 0; --bb) {
                Sb[bb * DK + ch] = sp;
                sp *= a[bb] * bi[bb];
            }
            int row = 0;
#pragma unroll
            for (int R = 1; R <= 3; ++R) {  // M(b, R) for b = 2R-1 .. 0
                float m = a[2 * R];
#pragma unroll
                for (int bb = 2 * R - 1; bb >= 0; --bb) {
                    Mt[(row + bb) * DK + ch] = m;
                    m *= bi[bb] * a[bb];
                }
                row += 2 * R;
            }
        }
        __syncthreads();
        // (c) per (block, channel pair): local products (packed fp32x2), then every
        //     operand row, two adjacent channels per 32-bit store
        for (int e = tid; e < 8 * (DK / 2); e += kThreads) {
            const int bb = e / (DK / 2), ch = 2 * (e % (DK / 2));
            const int r0 = 8 * bb;
            float2 al[8], kq[8], qq[8], f[8], gq[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                al[u] = *reinterpret_cast<const float2*>(&sm.al[(r0 + u) * DK + ch]);
                kq[u] = *reinterpret_cast<const float2*>(&sm.kn[(r0 + u) * DK + ch]);
                qq[u] = scale2(ld2(&sm.qr[(r0 + u) * DK + ch]), sm.iq[r0 + u]);
            }
            f[0] = make_float2(1.f, 1.f);
#pragma unroll
            for (int u = 1; u < 8; ++u) f[u] = mul2(f[u - 1], al[u]);
            gq[7] = make_float2(1.f, 1.f);
#pragma unroll
            for (int u = 6; u >= 0; --u) gq[u] = mul2(gq[u + 1], al[u + 1]);
            const float2 gb = *reinterpret_cast<const float2*>(&Gb[bb * DK + ch]);
            // QG = qh * gamma (global, operand layout); KT is formed in P6
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float2 qgv = mul2(qq[u], mul2(gb, f[u]));
                *reinterpret_cast<uint32_t*>(&gWQ[op_index_rm(kChunk + r0 + u, ch, DK)]) = pack_bf16(qgv.x, qgv.y);
            }
            const int R = bb >> 1;
            if (bb >= 2) {  // 16-level row factors D(r, 16R)
                float2 pre = make_float2(1.f, 1.f);
                if (bb & 1)
                    pre = mul2(*reinterpret_cast<const float2*>(&Bi[(2 * R) * DK + ch]),
                               *reinterpret_cast<const float2*>(&sm.al[(16 * R + 8) * DK + ch]));
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int rr = r0 + u - 16;
                    const float2 pf = mul2(pre, f[u]);
                    const float2 x = mul2(kq[u], pf), y = mul2(qq[u], pf);
                    *reinterpret_cast<uint32_t*>(&sm.ops.m.left[sw<DK>(rr, ch)]) = pack_bf16(x.x, x.y);
                    *reinterpret_cast<uint32_t*>(&sm.ops.m.leftq[sw<DK>(rr, ch)]) = pack_bf16(y.x, y.y);
                }
            }
            if (bb & 1) {  // 8-level row factors D(r, 16R+8)
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float2 x = mul2(kq[u], f[u]), y = mul2(qq[u], f[u]);
                    *reinterpret_cast<uint32_t*>(&sm.ops.m.l8[sw<DK>(8 * R + u, ch)]) = pack_bf16(x.x, x.y);
                    *reinterpret_cast<uint32_t*>(&sm.ops.m.l8q[sw<DK>(8 * R + u, ch)]) = pack_bf16(y.x, y.y);
                }
            } else {       // 8-level column factors D(16R+8, j) = g_j alpha(16R+8)
                const float2 a8 = *reinterpret_cast<const float2*>(&sm.al[(16 * R + 8) * DK + ch]);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float2 x = mul2(kq[u], mul2(gq[u], a8));
                    *reinterpret_cast<uint32_t*>(&sm.ops.m.r8[sw<DK>(8 * R + u, ch)]) = pack_bf16(x.x, x.y);
                }
            }
            // 16-level column factors D(16R', j) for every R' with 16R' > j
            int mrow = 0, rbase = 0;
#pragma unroll
            for (int Rp = 1; Rp <= 3; ++Rp) {
                if (bb < 2 * Rp) {
                    const float2 m = *reinterpret_cast<const float2*>(&Mt[(mrow + bb) * DK + ch]);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float2 x = mul2(kq[u], mul2(gq[u], m));
                        *reinterpret_cast<uint32_t*>(&sm.ops.m.right[sw<DK>(rbase + r0 + u, ch)]) =
                            pack_bf16(x.x, x.y);
                    }
                }
                mrow += 2 * Rp;
                rbase += 16 * Rp;
            }
        }
        (void)TPB;
    }
    __syncthreads();

    // ------------------------------------------ P3: factorised blocks on mma.sync
    // Warps 0-11: one 8-column tile each of the 16-level blocks (R = 1: 2 tiles,
    // R = 2: 4, R = 3: 6), A and P together.  Warps 12-15: the 8 x 8 quadrant of
    // diagonal 16-block R = warp - 12.
    {
        const int gq = lane >> 2, tq = lane & 3;
        if (warp < 12) {
            const int R = warp < 2 ? 1 : (warp < 6 ? 2 : 3);
            const int nt = warp < 2 ? warp : (warp < 6 ? warp - 2 : warp - 6);
            const int rbase = (R - 1) * 16;                    // rows in left/leftq
            const int cbase = R == 1 ? 0 : (R == 2 ? 16 : 48); // rows in right
            float accA[4] = {0.f, 0.f, 0.f, 0.f}, accP[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const int k0 = kk * 16 + 2 * tq;
                uint32_t a[4], aq[4];
                a[0] = lds_pair<DK>(sm.ops.m.left, rbase + gq, k0);
                a[1] = lds_pair<DK>(sm.ops.m.left, rbase + gq + 8, k0);
                a[2] = lds_pair<DK>(sm.ops.m.left, rbase + gq, k0 + 8);
                a[3] = lds_pair<DK>(sm.ops.m.left, rbase + gq + 8, k0 + 8);
                aq[0] = lds_pair<DK>(sm.ops.m.leftq, rbase + gq, k0);
                aq[1] = lds_pair<DK>(sm.ops.m.leftq, rbase + gq + 8, k0);
                aq[2] = lds_pair<DK>(sm.ops.m.leftq, rbase + gq, k0 + 8);
                aq[3] = lds_pair<DK>(sm.ops.m.leftq, rbase + gq + 8, k0 + 8);
                const int brow = cbase + nt * 8 + gq;
                const uint32_t b0 = lds_pair<DK>(sm.ops.m.right, brow, k0);
                const uint32_t b1 = lds_pair<DK>(sm.ops.m.right, brow, k0 + 8);
                mma16816(accA, a, b0, b1);
                mma16816(accP, aq, b0, b1);
            }
            const int col = nt * 8 + 2 * tq;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = 16 * R + gq + 8 * hh;
                const float b = sm.bs[row];
                sm.A[row * AP + col] = b * accA[2 * hh];
                sm.A[row * AP + col + 1] = b * accA[2 * hh + 1];
                *reinterpret_cast<uint32_t*>(&gP[op_index(row, col, kChunk)]) =
                    pack_bf16(accP[2 * hh], accP[2 * hh + 1]);
            }
        } else {
            // 8-level quadrant of diagonal block R: rows 16R+8.., cols 16R..
            const int R = warp - 12;
            float accA[4] = {0.f, 0.f, 0.f, 0.f}, accP[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                const int k0 = kk * 16 + 2 * tq;
                uint32_t a[4], aq[4];
                a[0] = lds_pair<DK>(sm.ops.m.l8, 8 * R + gq, k0);
                a[2] = lds_pair<DK>(sm.ops.m.l8, 8 * R + gq, k0 + 8);
                aq[0] = lds_pair<DK>(sm.ops.m.l8q, 8 * R + gq, k0);
                aq[2] = lds_pair<DK>(sm.ops.m.l8q, 8 * R + gq, k0 + 8);
                a[1] = a[3] = aq[1] = aq[3] = 0u;  // fragment rows 8-15 unused
                const uint32_t b0 = lds_pair<DK>(sm.ops.m.r8, 8 * R + gq, k0);
                const uint32_t b1 = lds_pair<DK>(sm.ops.m.r8, 8 * R + gq, k0 + 8);
                mma16816(accA, a, b0, b1);
                mma16816(accP, aq, b0, b1);
            }
            const int row = 16 * R + 8 + gq, col = 16 * R + 2 * tq;
            const float b = sm.bs[row];
            sm.A[row * AP + col] = b * accA[0];
            sm.A[row * AP + col + 1] = b * accA[1];
            *reinterpret_cast<uint32_t*>(&gP[op_index(row, col, kChunk)]) = pack_bf16(accP[0], accP[1]);
            // zero blocks of P above the diagonal, whole 8 x 8 core matrices (128
            // contiguous bytes each): the upper-right quadrant of diagonal block R
            // and the 16 x 16 blocks (R, J > R)
            uint4* gP4 = reinterpret_cast<uint4*>(gP);
            const uint4 z4 = make_uint4(0, 0, 0, 0);
            if (lane < 8) gP4[op_index(16 * R, 16 * R + 8, kChunk) / 8 + lane] = z4;
            for (int J = R + 1; J < 4; ++J)  // core matrices (2R + i, 2J + c), 8 words each
                gP4[op_index(16 * R + 8 * (lane >> 4), 16 * J + 8 * ((lane >> 3) & 1), kChunk) / 8 +
                    (lane & 7)] = z4;
        }
    }

    // ------------------------------------- P4: 8 x 8 diagonal blocks (CUDA cores)
    // Thread (block, row pair {a, 7 - a}, group of DK/16 channels): row a has a + 1
    // entries on or below the diagonal and row 7 - a has 8 - a, so every lane runs
    // the same 9 steps.  Channel pairs use packed fp32x2 arithmetic; their order is
    // rotated so that a warp's 64-bit shared loads take two wavefronts.  The two
    // warps of a block each cover half of the channels and meet in shared memory.
    {
        constexpr int CG = DK / 16, CPp = CG / 2;
        const int blk = warp >> 1, half = warp & 1;
        const int rp = lane >> 3, cg = (lane & 7) + 8 * half;
        const int ra = 8 * blk + rp, rz = 8 * blk + 7 - rp;
        float2 acc2A[9], acc2P[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) acc2A[t] = acc2P[t] = make_float2(0.f, 0.f);
        const float iqa = sm.iq[ra], iqz = sm.iq[rz];
#pragma unroll 1
        for (int i = 0; i < CPp; ++i) {
            const int ch = cg * CG + 2 * ((i + 2 * ((lane >> 2) & 1) + rp) & (CPp - 1));
            const float2 ka = *reinterpret_cast<const float2*>(&sm.kn[ra * DK + ch]);
            const float2 qa = scale2(ld2(&sm.qr[ra * DK + ch]), iqa);
            const float2 kz = *reinterpret_cast<const float2*>(&sm.kn[rz * DK + ch]);
            const float2 qz = scale2(ld2(&sm.qr[rz * DK + ch]), iqz);
            float2 f = make_float2(1.f, 1.f);
#pragma unroll
            for (int t = 0; t < 9; ++t) {
                const bool first = t <= rp;
                const int j = first ? ra - t : 8 * blk + 8 - t;
                if (t == 0 || t == rp + 1) {
                    f = make_float2(1.f, 1.f);
                } else {
                    f = mul2(f, *reinterpret_cast<const float2*>(&sm.al[(j + 1) * DK + ch]));
                }
                const float2 tk = mul2(*reinterpret_cast<const float2*>(&sm.kn[j * DK + ch]), f);
                acc2P[t] = fma2(first ? qa : qz, tk, acc2P[t]);
                acc2A[t] = fma2(first ? ka : kz, tk, acc2A[t]);
            }
        }
        float accA[9], accP[9];
#pragma unroll
        for (int t = 0; t < 9; ++t) {
            accA[t] = acc2A[t].x + acc2A[t].y;
            accP[t] = acc2P[t].x + acc2P[t].y;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                accA[t] += __shfl_xor_sync(0xffffffffu, accA[t], o);
                accP[t] += __shfl_xor_sync(0xffffffffu, accP[t], o);
            }
        }
        float* part = sm.X + (blk * 4 + rp) * 18;  // X is free until the inverse
        if (half == 1 && (lane & 7) == 0) {
#pragma unroll
            for (int t = 0; t < 9; ++t) {
                part[t] = accA[t];
                part[9 + t] = accP[t];
            }
        }
        __syncthreads();
        if (half == 0) {
            // The 8 lanes of a group hold the same totals; lane j stores entry t = j
            // (lane 0 also t = 8) of A into shared memory and column 8 blk + j of the
            // group's two P rows (one 16-byte run per row across the group).
            const int j8 = lane & 7, g0 = lane & ~7;
            const float ba = sm.bs[ra], bz = sm.bs[rz];
            auto entry = [&](int t, float aA, float aP) {
                const bool first = t <= rp;
                const int r = first ? ra : rz;
                const int jc = first ? ra - t : 8 * blk + 8 - t;
                if (jc < r) sm.A[r * AP + jc] = (first ? ba : bz) * (aA + part[t]);
                return aP + part[9 + t];
            };
            float aA = accA[0], aP = accP[0];
#pragma unroll
            for (int t = 1; t < 8; ++t)
                if (j8 == t) { aA = accA[t]; aP = accP[t]; }
            const float pv = entry(j8, aA, aP);
            const float pv8 = j8 == 0 ? entry(8, accA[8], accP[8]) : 0.f;
            // row rz, column 8 blk + u needs t = 8 - u (u <= 7 - rp); row ra needs t = rp - u
            const float z8 = __shfl_sync(0xffffffffu, pv8, g0);
            const float zt = __shfl_sync(0xffffffffu, pv, g0 | ((8 - j8) & 7));
            const float at = __shfl_sync(0xffffffffu, pv, g0 | ((rp - j8) & 7));
            const float pz = j8 <= 7 - rp ? (j8 == 0 ? z8 : zt) : 0.f;
            const float pa = j8 <= rp ? at : 0.f;
            gP[op_index(ra, 8 * blk + j8, kChunk)] = __float2bfloat16(pa);
            gP[op_index(rz, 8 * blk + j8, kChunk)] = __float2bfloat16(pz);
        }
    }
    ptx::fence_proxy_async_smem();  // reads of qn above come before the copy into it
    __syncthreads();

    if (kBf16In && tid == 0 && next.h < H) issue_q(next, rows_next);

    // ------------------------------------- P5: X = (I + A)^-1 by recursive doubling
    // 8 x 8 diagonal blocks by forward substitution (written whole, zeros above the
    // diagonal), then for n = 8, 16, 32: X21 = -X22 (A21 X11) joins two inverted n x n
    // blocks into one 2n x 2n block (n = 8 on CUDA cores, n = 16 and 32 with mma.sync
    // on tf32 inputs and fp32 accumulation).  Entries of X above the diagonal are never
    // written; the joins read them as zero, and nothing else reads them.
    {
        if (tid < 64) {
            const int base = 8 * (tid >> 3), jc = tid & 7;
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float acc = (i == jc) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m < i) acc -= sm.A[(base + i) * AP + base + m] * x[m];
                x[i] = (i < jc) ? 0.f : acc;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) sm.X[(base + i) * AP + base + jc] = x[i];
        }
        __syncthreads();
        inv_join<8>(sm.X, sm.A, sm.ops.scratch, tid);
        inv_join_tc<16>(sm.X, sm.A, sm.ops.scratch, warp, lane);
        inv_join_tc<32>(sm.X, sm.A, sm.ops.scratch, warp, lane);
    }

    // ------------------------------------- P6: tcgen05 operands X Diag(beta), [kh g | v]^T
    {
        for (int e = tid; e < kChunk * 8; e += kThreads) {
            const int i = e >> 3, jb = (e & 7) * 8;
            float x[8], lo[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = jb + u;
                x[u] = (j <= i) ? sm.X[i * AP + j] * sm.bs[j] : 0.f;
            }
            const uint4 hi = pack8(x);
            const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hi);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                lo[2 * u] = x[2 * u] - f.x;
                lo[2 * u + 1] = x[2 * u + 1] - f.y;
            }
            *reinterpret_cast<uint4*>(&sm.ops.t.xop[op_index(i, jb, kChunk)]) = hi;
            *reinterpret_cast<uint4*>(&sm.ops.t.xlo[op_index(i, jb, kChunk)]) = pack8(lo);
        }
        // [kh * gamma | v]^T, one task per (8-row block, column): gamma_r = Gb_b f_r
        // k columns and v columns in separate loops, so every thread gets its share of
        // the heavier k tasks
        for (int e = tid; e < 8 * DK; e += kThreads) {
            const int bb = e / DK, col = e % DK, r0 = 8 * bb;
            {
                // gamma_r = Gb_b * alpha(r0+1..r) and gamma_L / gamma_r = alpha(r+1..r0+7) * Sb_b
                float a[8], kv[8], x[8], kt[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    a[u] = sm.al[(r0 + u) * DK + col];
                    kv[u] = sm.kn[(r0 + u) * DK + col];
                }
                float f = sm.gb[bb * DK + col], bk = sm.sb[bb * DK + col];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (u > 0) f *= a[u];
                    x[u] = kv[u] * f;
                }
#pragma unroll
                for (int u = 7; u >= 0; --u) {
                    kt[u] = kv[u] * bk;
                    bk *= a[u];
                }
                *reinterpret_cast<uint4*>(&sm.ops.t.bop[op_index(col, r0, NB)]) = pack8(x);
                // KT (fp32, tf32 operand layout): rows r0..r0+7 are two 16-byte runs
                float* kth = r0 < kChunk / 2 ? st_kt0 : st_kt1 - KTH;  // rows 0-31 | 32-63
                *reinterpret_cast<float4*>(&kth[op_index32(col, r0, DK)]) = make_float4(kt[0], kt[1], kt[2], kt[3]);
                *reinterpret_cast<float4*>(&kth[op_index32(col, r0 + 4, DK)]) = make_float4(kt[4], kt[5], kt[6], kt[7]);
            }
        }
        for (int e = tid; e < 8 * DV; e += kThreads) {
            const int bb = e / DV, dcol = e % DV, r0 = 8 * bb;
            uint4 u4;
            __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(&u4);
#pragma unroll
            for (int u = 0; u < 8; ++u) hb[u] = sm.vs[(r0 + u) * DV + dcol];
            *reinterpret_cast<uint4*>(&sm.ops.t.bop[op_index(DK + dcol, r0, NB)]) = u4;
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    // ------------------------------------------------- P7: [w | u] on tcgen05
    if (tid == 0) {
        // X Diag(beta) = hi + lo (both bf16): the split keeps the inverse's fp32
        // accuracy through the product
        const uint32_t ba = ptx::smem_u32(sm.ops.t.bop);
        constexpr uint32_t idesc = ptx::idesc_bf16(kChunk, NB);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const uint32_t xa = ptx::smem_u32(part ? sm.ops.t.xlo : sm.ops.t.xop);
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
                ptx::mma_bf16(tmem, ptx::smem_desc(xa + kk * 2048, 1024, 128),
                              ptx::smem_desc(ba + kk * 2 * (NB / 8) * 128, (NB / 8) * 128, 128),
                              idesc, part > 0 || kk > 0);
        }
        ptx::mma_commit(&sm.bar);
        // KT leaves by bulk copies (rows 0-31 and 32-63 of the chunk are the two
        // contiguous halves of its operand layout)
        ptx::bulk_s2g(gKT, st_kt0, KTH * 4);
        ptx::bulk_s2g(gKT + KTH, st_kt1, KTH * 4);
        ptx::bulk_commit();
        if (!kBf16In) ptx::bulk_wait_read_all();  // fp32 inputs land where KT was staged
        if (next.h < H) {  // lands while the epilogue runs
            if (kBf16In) issue_kgv(next, rows_next);
            else issue_copies(next, rows_next);
        }
    }
    if (next.h < H) load_beta(next, rows_next);
    const bool ok = ptx::mbar_wait_or_abort(&sm.bar, phase, &sm.abort);
    if (!ok && tid == 0) atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
    ptx::tc_fence_after();
    {
        // warps w, w + 4, w + 8, w + 12 share TMEM lane quarter w; split the columns.
        // The results are staged in shared memory (the operand region, dead once the
        // MMA has completed) in their global layouts and leave by bulk copies.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = 16 * quarter + lane;  // valid for lane < 16 (M = 64 layout)
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        constexpr int HALF = NB / (kThreads / 128), NLD = HALF / 16;
        float x[NLD][16];  // all of this warp's columns, then one wait
#pragma unroll
        for (int i = 0; i < NLD; ++i) ptx::tmem_ld16(tmem + lane_base + half * HALF + 16 * i, x[i]);
        ptx::tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 2 * NLD; ++i) {
                const int col = half * HALF + 8 * i;
                float y[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) y[u] = x[i >> 1][8 * (i & 1) + u];
                if (col < DK) {  // w: rows 0-63 of the 128-row tile, one contiguous block
                    *reinterpret_cast<uint4*>(&st_w[op_index_rm(row, col, DK)]) = pack8(y);
                } else {         // u stays fp32
                    const int n = col - DK;
                    *reinterpret_cast<float4*>(&st_u[u0_index(row, n)]) = make_float4(y[0], y[1], y[2], y[3]);
                    *reinterpret_cast<float4*>(&st_u[u0_index(row, n + 4)]) = make_float4(y[4], y[5], y[6], y[7]);
                }
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        ptx::bulk_s2g(gWQ, st_w, kChunk * DK * 2);  // w: the first half of the WQ tile
        ptx::bulk_s2g(gU, st_u, kChunk * DV * 4);
        ptx::bulk_commit();
    }
    ptx::tc_fence_after();
    phase ^= 1u;
    item = next;
    rows_cur = rows_next;
    }  // items
    if (tid == 0) ptx::bulk_wait_all();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

// The driver's tensor-map encoder, fetched once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Tensor map of a [tokens, H, D] row-major tensor with a box of 64 tokens x 1 head
// x D channels (so one copy brings one chunk of one head).
bool encode_rows(CUtensorMap* m, const void* base, bool f32, int D, int H, long long tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {D * es, (cuuint64_t)H * D * es};
    const cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)kChunk};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV, typename TIn, typename TG>
cudaError_t launch_t(const Dims& d, const void* q, const void* k, const void* v, const void* g,
                     const float* beta, uint8_t* ws, cudaStream_t stream) {
    auto kern = prep_tc_kernel<DK, DV, TIn, TG>;
    const size_t smem = sizeof(PrepSmem<DK, DV, TIn>);
    const WsLayout W(d);
    const long long tokens = (long long)d.B * d.T;
    if (W.cmax == 0 || tokens == 0) return cudaSuccess;  // no chunk has a token
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    constexpr bool f32 = sizeof(TIn) == 4;
    CUtensorMap tq, tk, tv, tg;
    if (!encode_rows(&tq, q, f32, DK, d.H, tokens) || !encode_rows(&tk, k, f32, DK, d.H, tokens) ||
        !encode_rows(&tv, v, f32, DV, d.H, tokens) || !encode_rows(&tg, g, sizeof(TG) == 4, DK, d.H, tokens))
        return cudaErrorInvalidValue;
    const long long items = W.cmax * d.H;
    const unsigned grid = (unsigned)(items < num_sms() ? items : num_sms());  // persistent
    kern<<<grid, kThreads, smem, stream>>>(d, tq, tk, tv, tg, beta, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const Dims& d, bool qkv_bf16, bool g_bf16, const void* q, const void* k,
                           const void* v, const void* g, const float* beta, uint8_t* ws,
                           cudaStream_t stream) {
    using bf = __nv_bfloat16;
#define KDA_PREP_CASE(DK_, DV_)                                                                  \
    if (d.dk == DK_ && d.dv == DV_) {                                                            \
        if (!qkv_bf16) return g_bf16 ? cudaErrorInvalidValue                                     \
                                     : launch_t<DK_, DV_, float, float>(d, q, k, v, g, beta, ws, stream); \
        return g_bf16 ? launch_t<DK_, DV_, bf, bf>(d, q, k, v, g, beta, ws, stream)               \
                      : launch_t<DK_, DV_, bf, float>(d, q, k, v, g, beta, ws, stream);           \
    }
    KDA_PREP_CASE(64, 64)
    KDA_PREP_CASE(64, 128)
    KDA_PREP_CASE(128, 64)
    KDA_PREP_CASE(128, 128)
#undef KDA_PREP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
