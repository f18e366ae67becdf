// Factor kernel of the three-kernel pipeline: the factor body (kda_factor_body.cuh)
// over head-major (chunk, head) items in steps of the grid size; the tensor maps of
// the inputs; the launcher.
#include "kda_factor_body.cuh"

namespace kda {

namespace {

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

}  // namespace

// Tensor map of a [tokens, H, D] row-major tensor with a box of 64 tokens x 1 head
// x D channels (one copy brings one chunk of one head, rows in order).
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

// Tensor map of a bf16 [tokens, H, D] tensor seen as {8 channels, tokens, H, D/8
// channel groups} (strides: a token row, a head, 16 bytes), with a box of 8 x 64
// tokens x 1 x D/8: one copy lands a chunk of one head as [D/8][64 rows][8], the
// N-major core-matrix layout of a tensor-core operand.
bool encode_groups(CUtensorMap* m, const void* base, int D, int H, long long tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {8, (cuuint64_t)tokens, (cuuint64_t)H, (cuuint64_t)(D / 8)};
    const cuuint64_t strides[3] = {(cuuint64_t)H * D * 2, (cuuint64_t)D * 2, 16};
    const cuuint32_t box[4] = {8, (cuuint32_t)kChunk, 1, (cuuint32_t)(D / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int DK, int DV, typename TIn, typename TG>
__global__ void __launch_bounds__(kThreads, 1)
    factor_kernel(Dims d, const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                  const float* __restrict__ beta, uint8_t* __restrict__ ws) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-column chain kernel and the segment passes, when they run, read u in
    // their own layout
    const Header* hdr = reinterpret_cast<const Header*>(ws + WsLayout(d).header);
    const bool ut = DK == 128 && DV == 128 && (hdr->chain128 || hdr->seg);
    factor_body<DK, DV, TIn, TG>(d, &tm_q, &tm_k, &tm_v, &tm_g, beta, ws, smem_raw,
                                 ItemPlan{nullptr, (int)blockIdx.x, (int)gridDim.x, nullptr, ut});
}

template <int DK, int DV, typename TIn, typename TG>
cudaError_t launch_t(const Dims& d, const void* q, const void* k, const void* v, const void* g,
                     const float* beta, uint8_t* ws, cudaStream_t stream) {
    using Sm = FactorSmem<DK, DV, TIn>;
    static_assert(sizeof(Sm) <= 227 * 1024, "factor kernel shared memory");
    static_assert(offsetof(Sm, qr) % 128 == 0 && offsetof(Sm, kr) % 128 == 0 &&
                      offsetof(Sm, gr) % 128 == 0 && offsetof(Sm, vs) % 128 == 0 &&
                      offsetof(Sm, kg) % 128 == 0,
                  "tensor-copy and operand destinations are 128-byte aligned");
    auto kern = factor_kernel<DK, DV, TIn, TG>;
    const size_t smem = sizeof(Sm);
    const WsLayout W(d);
    const long long tokens = (long long)d.B * d.T;
    if (W.cmax == 0 || tokens == 0) return cudaSuccess;  // no chunk has a token
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    constexpr bool f32 = sizeof(TIn) == 4;
    CUtensorMap tq, tk, tv, tg;
    const bool okv = f32 ? encode_rows(&tv, v, true, DV, d.H, tokens) : encode_groups(&tv, v, DV, d.H, tokens);
    if (!encode_rows(&tq, q, f32, DK, d.H, tokens) || !encode_rows(&tk, k, f32, DK, d.H, tokens) || !okv ||
        !encode_rows(&tg, g, sizeof(TG) == 4, DK, d.H, tokens))
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
#define KDA_FACTOR_CASE(DK_, DV_)                                                                 \
    if (d.dk == DK_ && d.dv == DV_) {                                                             \
        if (!qkv_bf16) return g_bf16 ? cudaErrorInvalidValue                                      \
                                     : launch_t<DK_, DV_, float, float>(d, q, k, v, g, beta, ws, stream); \
        return g_bf16 ? launch_t<DK_, DV_, bf, bf>(d, q, k, v, g, beta, ws, stream)                \
                      : launch_t<DK_, DV_, bf, float>(d, q, k, v, g, beta, ws, stream);            \
    }
    KDA_FACTOR_CASE(64, 64)
    KDA_FACTOR_CASE(64, 128)
    KDA_FACTOR_CASE(128, 64)
    KDA_FACTOR_CASE(128, 128)
#undef KDA_FACTOR_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda
