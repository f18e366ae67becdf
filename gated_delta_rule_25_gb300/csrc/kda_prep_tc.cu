// Per-chunk factors of the chunkwise KDA forward on tensor cores: one CTA per
// (chunk, head), 256 threads.
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
//   [w | u]  = X Diag(beta) [kh * gamma | v]                     (tcgen05, M=64 N=dk+dv K=64)
//   QG = qh * gamma,  KT = (kh * gamma_L / gamma)^T,  GL = gamma_L,  gamma = exp(Gamma)
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
#include "kda_internal.cuh"
#include "sm103_ptx.cuh"

namespace kda {

namespace {

constexpr int kThreads = 256;

template <int DK, int DV>
struct __align__(128) PrepSmem {
    float qn[kChunk * DK];
    float kn[kChunk * DK];
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
        struct {
            __nv_bfloat16 xop[kChunk * kChunk];        // X Diag(beta), operand layout
            __nv_bfloat16 bop[(DK + DV) * kChunk];     // [kh*gamma | v]^T, operand layout
        } t;
        float scratch[3 * 16 * 16];
    } ops;
    float bs[kChunk];
    uint64_t bar;
    uint32_t tmem;
    int abort;
};

template <typename TIn>
__device__ inline void load8(const TIn* p, float (&x)[8]);
template <>
__device__ inline void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
template <>
__device__ inline void load8<float>(const float* p, float (&x)[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

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

__device__ inline void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(kThreads, 1)
    prep_tc_kernel(Dims d, const TIn* __restrict__ q, const TIn* __restrict__ k,
                   const TIn* __restrict__ v, const float* __restrict__ g,
                   const float* __restrict__ beta, uint8_t* __restrict__ ws) {
    using Sm = PrepSmem<DK, DV>;
    constexpr int AP = kChunk + 1;
    constexpr int NB = DK + DV;  // columns of the w/u product
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    const WsLayout W(d);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= hdr->total_chunks) return;
    const int4 chk = reinterpret_cast<const int4*>(ws + W.chunks)[c];
    const long long row0 = chk.y;
    const int L = chk.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = d.H;
    const FactorLayout F(DK, DV);
    uint8_t* fb = ws + W.factors + ((size_t)c * H + h) * W.factor_bytes;
    __nv_bfloat16* gW = reinterpret_cast<__nv_bfloat16*>(fb + F.w);
    __nv_bfloat16* gQG = reinterpret_cast<__nv_bfloat16*>(fb + F.qg);
    __nv_bfloat16* gKT = reinterpret_cast<__nv_bfloat16*>(fb + F.kt);
    __nv_bfloat16* gP = reinterpret_cast<__nv_bfloat16*>(fb + F.p);
    __nv_bfloat16* gU = reinterpret_cast<__nv_bfloat16*>(fb + F.u0);
    float* gGL = reinterpret_cast<float*>(fb + F.gl);

    if (tid == 0) {
        ptx::mbar_init(&sm.bar, 1);
        sm.abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sm.tmem, 256);
        ptx::tmem_relinquish();
    }

    // ---------------------------------------------------------------- P1: load
    // 16-byte chunks: consecutive lanes take consecutive chunks of a row, so the
    // shared-memory stores are conflict free and a row's lanes reduce its norm.
    {
        constexpr int CPR = DK / 8;            // chunks per row
        constexpr int RP = kThreads / CPR;     // rows per pass
        const int ck = tid % CPR, rsub = tid / CPR;
#pragma unroll 1
        for (int r = rsub; r < kChunk; r += RP) {
            const bool valid = r < L;
            const size_t off = ((size_t)(row0 + r) * H + h) * DK + ck * 8;
            float xq[8], xk[8], xg[8];
            if (valid) {
                load8<TIn>(q + off, xq);
                load8<TIn>(k + off, xk);
                load8<float>(g + off, xg);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xq[e] = xk[e] = xg[e] = 0.f;
            }
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
            const float iq = rsqrtf(sq + 1e-6f), ik = rsqrtf(sk + 1e-6f);
            float* dq = &sm.qn[r * DK + ck * 8];
            float* dk_ = &sm.kn[r * DK + ck * 8];
            float* da = &sm.al[r * DK + ck * 8];
            *reinterpret_cast<float4*>(dq) = make_float4(xq[0] * iq, xq[1] * iq, xq[2] * iq, xq[3] * iq);
            *reinterpret_cast<float4*>(dq + 4) = make_float4(xq[4] * iq, xq[5] * iq, xq[6] * iq, xq[7] * iq);
            *reinterpret_cast<float4*>(dk_) = make_float4(xk[0] * ik, xk[1] * ik, xk[2] * ik, xk[3] * ik);
            *reinterpret_cast<float4*>(dk_ + 4) = make_float4(xk[4] * ik, xk[5] * ik, xk[6] * ik, xk[7] * ik);
            *reinterpret_cast<float4*>(da) = make_float4(__expf(xg[0]), __expf(xg[1]), __expf(xg[2]), __expf(xg[3]));
            *reinterpret_cast<float4*>(da + 4) = make_float4(__expf(xg[4]), __expf(xg[5]), __expf(xg[6]), __expf(xg[7]));
        }
        constexpr int VPR = DV / 8;
        constexpr int VRP = kThreads / VPR;
        const int vk = tid % VPR, vsub = tid / VPR;
#pragma unroll 1
        for (int r = vsub; r < kChunk; r += VRP) {
            float xv[8];
            if (r < L) load8<TIn>(v + ((size_t)(row0 + r) * H + h) * DV + vk * 8, xv);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[e] = 0.f;
            }
            *reinterpret_cast<uint4*>(&sm.vs[r * DV + vk * 8]) = pack8(xv);
        }
        if (tid < kChunk) sm.bs[tid] = tid < L ? beta[(size_t)(row0 + tid) * H + h] : 0.f;
    }
    __syncthreads();

    // ------------------------------------------------ P2: decay products per channel
    if (tid < DK) {
        // forward: gamma prefix (QG, GL), row factors of the mma operands
        const int ch = tid;
        float gp = 1.f, p16 = 1.f, p8 = 1.f;
        for (int r = 0; r < kChunk; ++r) {
            const float a = sm.al[r * DK + ch];
            gp *= a;
            const int ri = r & 15;
            p16 = ri == 0 ? 1.f : p16 * a;
            p8 = ri == 8 ? 1.f : p8 * a;
            const float kq = sm.kn[r * DK + ch], qq = sm.qn[r * DK + ch];
            if (r >= 16) {
                sm.ops.m.left[sw<DK>(r - 16, ch)] = __float2bfloat16(kq * p16);
                sm.ops.m.leftq[sw<DK>(r - 16, ch)] = __float2bfloat16(qq * p16);
            }
            if (ri >= 8) {
                const int rr = (r >> 4) * 8 + (ri - 8);
                sm.ops.m.l8[sw<DK>(rr, ch)] = __float2bfloat16(kq * p8);
                sm.ops.m.l8q[sw<DK>(rr, ch)] = __float2bfloat16(qq * p8);
            }
            gQG[op_index(r, ch, kChunk)] = __float2bfloat16(qq * gp);
        }
        gGL[ch] = gp;
    } else if (tid < 2 * DK) {
        // backward: suffix products (KT), column factors of the mma operands
        const int ch = tid - DK;
        float suf = 1.f;
        for (int rb = kChunk - 8; rb >= 0; rb -= 8) {
            float x[8];
#pragma unroll
            for (int e = 7; e >= 0; --e) {
                const int r = rb + e;
                x[e] = sm.kn[r * DK + ch] * suf;
                suf *= sm.al[r * DK + ch];
            }
            *reinterpret_cast<uint4*>(&gKT[op_index(ch, rb, DK)]) = pack8(x);
        }
        // 16-level column factors: f_m(j) = D(m, j) for anchors m = 16, 32, 48
        float f16[16], f32[16], f48[16];
        {
            float f = 1.f;
#pragma unroll
            for (int j = 15; j >= 0; --j) { f *= sm.al[(j + 1) * DK + ch]; f16[j] = f; }
            f = 1.f;
#pragma unroll
            for (int j = 15; j >= 0; --j) { f *= sm.al[(j + 17) * DK + ch]; f32[j] = f; }
            f = 1.f;
#pragma unroll
            for (int j = 15; j >= 0; --j) { f *= sm.al[(j + 33) * DK + ch]; f48[j] = f; }
        }
        const float d1632 = f32[0], d3248 = f48[0];  // D(32, 16), D(48, 32)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float k0 = sm.kn[j * DK + ch], k1 = sm.kn[(j + 16) * DK + ch];
            const float k2 = sm.kn[(j + 32) * DK + ch];
            sm.ops.m.right[sw<DK>(j, ch)] = __float2bfloat16(k0 * f16[j]);                   // R=1
            sm.ops.m.right[sw<DK>(16 + j, ch)] = __float2bfloat16(k0 * f16[j] * d1632);       // R=2
            sm.ops.m.right[sw<DK>(32 + j, ch)] = __float2bfloat16(k1 * f32[j]);
            sm.ops.m.right[sw<DK>(48 + j, ch)] = __float2bfloat16(k0 * f16[j] * d1632 * d3248);  // R=3
            sm.ops.m.right[sw<DK>(64 + j, ch)] = __float2bfloat16(k1 * f32[j] * d3248);
            sm.ops.m.right[sw<DK>(80 + j, ch)] = __float2bfloat16(k2 * f48[j]);
        }
        // 8-level column factors: D(16R+8, j), j in [16R, 16R+8)
#pragma unroll
        for (int R = 0; R < 4; ++R) {
            float f = 1.f;
#pragma unroll
            for (int e = 7; e >= 0; --e) {
                const int j = 16 * R + e;
                f *= sm.al[(j + 1) * DK + ch];
                sm.ops.m.r8[sw<DK>(8 * R + e, ch)] = __float2bfloat16(sm.kn[j * DK + ch] * f);
            }
        }
    }
    __syncthreads();

    // ------------------------------------------ P3: factorised blocks on mma.sync
    {
        const int gq = lane >> 2, tq = lane & 3;
        if (warp < 4) {
            // 16-level: block row R, n-tiles [n0, n1) of the 16R columns left of it
            const int R = warp == 0 ? 1 : (warp == 1 ? 2 : 3);
            const int n0 = warp == 3 ? 3 : 0;
            const int n1 = warp == 0 ? 2 : (warp == 1 ? 4 : (warp == 2 ? 3 : 6));
            const int rbase = (R - 1) * 16;                    // rows in left/leftq
            const int cbase = R == 1 ? 0 : (R == 2 ? 16 : 48); // rows in right
            float accA[4][4], accP[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) accA[n][e] = accP[n][e] = 0.f;
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
#pragma unroll
                for (int n = 0; n < 4; ++n) {
                    if (n0 + n < n1) {
                        const int brow = cbase + (n0 + n) * 8 + gq;
                        const uint32_t b0 = lds_pair<DK>(sm.ops.m.right, brow, k0);
                        const uint32_t b1 = lds_pair<DK>(sm.ops.m.right, brow, k0 + 8);
                        mma16816(accA[n], a, b0, b1);
                        mma16816(accP[n], aq, b0, b1);
                    }
                }
            }
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                if (n0 + n < n1) {
                    const int col = (n0 + n) * 8 + 2 * tq;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int row = 16 * R + gq + 8 * hh;
                        const float b = sm.bs[row];
                        sm.A[row * AP + col] = b * accA[n][2 * hh];
                        sm.A[row * AP + col + 1] = b * accA[n][2 * hh + 1];
                        gP[op_index(row, col, kChunk)] = __float2bfloat16(accP[n][2 * hh]);
                        gP[op_index(row, col + 1, kChunk)] = __float2bfloat16(accP[n][2 * hh + 1]);
                    }
                }
            }
        } else {
            // 8-level quadrant of diagonal block R = warp - 4: rows 16R+8.., cols 16R..
            const int R = warp - 4;
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
            gP[op_index(row, col, kChunk)] = __float2bfloat16(accP[0]);
            gP[op_index(row, col + 1, kChunk)] = __float2bfloat16(accP[1]);
            // zero blocks of P above the diagonal: upper-right quadrant of diagonal
            // block R and the 16 x 16 blocks (R, J > R)
            const __nv_bfloat16 z = __float2bfloat16(0.f);
            for (int e = lane; e < 64; e += 32) {
                const int rr = 16 * R + (e >> 3), cc = 16 * R + 8 + (e & 7);
                gP[op_index(rr, cc, kChunk)] = z;
            }
            for (int J = R + 1; J < 4; ++J)
                for (int e = lane; e < 256; e += 32)
                    gP[op_index(16 * R + (e >> 4), 16 * J + (e & 15), kChunk)] = z;
        }
    }

    // ------------------------------------- P4: 8 x 8 diagonal blocks (CUDA cores)
    {
        constexpr int CQ = DK / 4;
        const int blk = warp, rin = (lane >> 2) & 7, qt = lane & 3;
        const int r = 8 * blk + rin;
        float accA[8], accP[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) accA[e] = accP[e] = 0.f;
        for (int i = 0; i < CQ; ++i) {
            const int ch = qt * CQ + ((i + lane) & (CQ - 1));
            const float kr = sm.kn[r * DK + ch], qr = sm.qn[r * DK + ch];
            float f = 1.f;
#pragma unroll
            for (int dd = 0; dd < 8; ++dd) {
                if (dd <= rin) {
                    const int j = r - dd;
                    if (dd > 0) f *= sm.al[(j + 1) * DK + ch];
                    const float t = sm.kn[j * DK + ch] * f;
                    accP[dd] = fmaf(qr, t, accP[dd]);
                    accA[dd] = fmaf(kr, t, accA[dd]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            accA[e] += __shfl_xor_sync(0xffffffffu, accA[e], 1);
            accA[e] += __shfl_xor_sync(0xffffffffu, accA[e], 2);
            accP[e] += __shfl_xor_sync(0xffffffffu, accP[e], 1);
            accP[e] += __shfl_xor_sync(0xffffffffu, accP[e], 2);
        }
        if (qt == 0) {
            const float b = sm.bs[r];
#pragma unroll
            for (int dd = 0; dd < 8; ++dd) {
                if (dd <= rin) {
                    const int j = r - dd;
                    if (dd > 0) sm.A[r * AP + j] = b * accA[dd];
                    gP[op_index(r, j, kChunk)] = __float2bfloat16(accP[dd]);
                }
            }
            const __nv_bfloat16 z = __float2bfloat16(0.f);
            for (int j = r + 1; j < 8 * blk + 8; ++j) gP[op_index(r, j, kChunk)] = z;
        }
    }
    __syncthreads();

    // ------------------------------------------------- P5: X = (I + A)^-1, blocked
    {
        float* X = sm.X;
        const float* A = sm.A;
        // (a) diagonal 16-blocks by forward substitution, thread per (block, column)
        if (tid < 64) {
            const int b = tid >> 4, jc = tid & 15, base = 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float s = (i == jc) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    if (m < i) s -= A[(base + i) * AP + base + m] * x[m];
                x[i] = (i < jc) ? 0.f : s;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) X[(base + i) * AP + base + jc] = x[i];
        }
        __syncthreads();
        // (b) blocks below the diagonal, by distance: X_RJ = -X_RR sum_K A_RK X_KJ
        float* T = sm.ops.scratch;
        for (int dist = 1; dist <= 3; ++dist) {
            const int nblk = 4 - dist;
            for (int e = tid; e < nblk * 256; e += kThreads) {
                const int R = dist + e / 256, J = R - dist, i = (e % 256) >> 4, j = e & 15;
                float s = 0.f;
                for (int K = J; K < R; ++K)
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        s += A[(16 * R + i) * AP + 16 * K + m] * X[(16 * K + m) * AP + 16 * J + j];
                T[e] = s;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += kThreads) {
                const int R = dist + e / 256, J = R - dist, i = (e % 256) >> 4, j = e & 15;
                float s = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    s -= X[(16 * R + i) * AP + 16 * R + m] * T[(e / 256) * 256 + m * 16 + j];
                X[(16 * R + i) * AP + 16 * J + j] = s;
            }
            __syncthreads();
        }
    }

    // ------------------------------------- P6: tcgen05 operands X Diag(beta), [kh g | v]^T
    {
        for (int e = tid; e < kChunk * 8; e += kThreads) {
            const int i = e >> 3, jb = (e & 7) * 8;
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = jb + u;
                x[u] = ((j >> 4) <= (i >> 4)) ? sm.X[i * AP + j] * sm.bs[j] : 0.f;
            }
            *reinterpret_cast<uint4*>(&sm.ops.t.xop[op_index(i, jb, kChunk)]) = pack8(x);
        }
        for (int col = tid; col < NB; col += kThreads) {
            if (col < DK) {
                float gp = 1.f;
                for (int jb = 0; jb < kChunk; jb += 8) {
                    float x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        gp *= sm.al[(jb + u) * DK + col];
                        x[u] = sm.kn[(jb + u) * DK + col] * gp;
                    }
                    *reinterpret_cast<uint4*>(&sm.ops.t.bop[op_index(col, jb, NB)]) = pack8(x);
                }
            } else {
                const int dcol = col - DK;
                for (int jb = 0; jb < kChunk; jb += 8) {
                    uint4 u4;
                    __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(&u4);
#pragma unroll
                    for (int u = 0; u < 8; ++u) hb[u] = sm.vs[(jb + u) * DV + dcol];
                    *reinterpret_cast<uint4*>(&sm.ops.t.bop[op_index(col, jb, NB)]) = u4;
                }
            }
        }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sm.tmem;

    // ------------------------------------------------- P7: [w | u] on tcgen05
    if (tid == 0) {
        const uint32_t xa = ptx::smem_u32(sm.ops.t.xop), ba = ptx::smem_u32(sm.ops.t.bop);
        constexpr uint32_t idesc = ptx::idesc_bf16(kChunk, NB);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
            ptx::mma_bf16(tmem, ptx::smem_desc(xa + kk * 2048, 1024, 128),
                          ptx::smem_desc(ba + kk * 2 * (NB / 8) * 128, (NB / 8) * 128, 128), idesc,
                          kk > 0);
        ptx::mma_commit(&sm.bar);
    }
    const bool ok = ptx::mbar_wait_or_abort(&sm.bar, 0, &sm.abort);
    if (!ok && tid == 0) atomicOr(reinterpret_cast<unsigned int*>(ws), kDevErrTimeout);
    ptx::tc_fence_after();
    {
        // warp w and w + 4 share TMEM lane quarter w; split the columns between them
        const int quarter = warp & 3, half = warp >> 2;
        const int row = 16 * quarter + lane;  // valid for lane < 16 (M = 64 layout)
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        constexpr int HALF = NB / 2;
#pragma unroll 1
        for (int cb = half * HALF; cb < (half + 1) * HALF; cb += 16) {
            float x[16];
            ptx::tmem_ld16(tmem + lane_base + cb, x);
            ptx::tmem_ld_wait();
            if (ok && lane < 16) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int col = cb + 8 * hh;
                    float y[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) y[u] = x[8 * hh + u];
                    if (col < DK)
                        *reinterpret_cast<uint4*>(&gW[op_index(row, col, kChunk)]) = pack8(y);
                    else
                        *reinterpret_cast<uint4*>(&gU[u0_index(row, col - DK)]) = pack8(y);
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 256);
    }
}

template <int DK, int DV, typename TIn>
cudaError_t launch_t(const Dims& d, const void* q, const void* k, const void* v, const float* g,
                     const float* beta, uint8_t* ws, cudaStream_t stream) {
    auto kern = prep_tc_kernel<DK, DV, TIn>;
    const size_t smem = sizeof(PrepSmem<DK, DV>);
    const WsLayout W(d);
    if (W.cmax == 0) return cudaSuccess;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)W.cmax, (unsigned)d.H);
    kern<<<grid, kThreads, smem, stream>>>(d, static_cast<const TIn*>(q), static_cast<const TIn*>(k),
                                           static_cast<const TIn*>(v), g, beta, ws);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_tc(const Dims& d, bool qkv_bf16, const void* q, const void* k,
                           const void* v, const float* g, const float* beta, uint8_t* ws,
                           cudaStream_t stream) {
#define KDA_PREP_CASE(DK_, DV_)                                                                   \
    if (d.dk == DK_ && d.dv == DV_)                                                               \
        return qkv_bf16 ? launch_t<DK_, DV_, __nv_bfloat16>(d, q, k, v, g, beta, ws, stream)       \
                        : launch_t<DK_, DV_, float>(d, q, k, v, g, beta, ws, stream);
    KDA_PREP_CASE(64, 64)
    KDA_PREP_CASE(64, 128)
    KDA_PREP_CASE(128, 64)
    KDA_PREP_CASE(128, 128)
#undef KDA_PREP_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
