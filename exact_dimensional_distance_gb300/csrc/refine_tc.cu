// Tensor-core (tcgen05) building blocks.
//
// gram_tf32: the Gram matrix G = A B^T of two 128-row float32 blocks after
// rounding both to TF32, computed by one CTA with tcgen05.mma (kind::tf32,
// M = N = 128, accumulator in tensor memory) from operands staged in shared
// memory in the no-swizzle K-major core-matrix layout.  It exercises the
// descriptors, the instruction descriptor and the tensor-memory layout that
// the tensor-core refinement uses.
#include "hiss_internal.cuh"
#include "ptx.cuh"

namespace hiss {
namespace {

constexpr int kGramRows = 128;

// Byte offset of element (row, k) of a K-major operand with kpad columns in
// the no-swizzle core-matrix layout: core matrices of 8 rows x 4 TF32
// elements (128 bytes) are contiguous along K (lbo = 128 bytes); groups of 8
// rows follow each other (sbo = kpad / 4 * 128 bytes).
__host__ __device__ __forceinline__ uint32_t core_offset(int row, int k, int kpad)
{
    return (uint32_t)((row >> 3) * (kpad / 4) * 128 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

__global__ void __launch_bounds__(128, 1) k_gram_tf32(const float *a, const float *b, int k, float *out, int *flags)
{
    extern __shared__ __align__(128) unsigned char gsm[];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned char *As = gsm;
    unsigned char *Bs = gsm + (size_t)kGramRows * k * 4;
    // row tid of both operands, TF32-rounded, into the core-matrix layout
    for (int kc = 0; kc < k / 4; ++kc) {
        const float4 va = *reinterpret_cast<const float4 *>(a + (int64_t)tid * k + 4 * kc);
        const float4 vb = *reinterpret_cast<const float4 *>(b + (int64_t)tid * k + 4 * kc);
        *reinterpret_cast<float4 *>(As + core_offset(tid, 4 * kc, k)) =
            make_float4(to_tf32(va.x), to_tf32(va.y), to_tf32(va.z), to_tf32(va.w));
        *reinterpret_cast<float4 *>(Bs + core_offset(tid, 4 * kc, k)) =
            make_float4(to_tf32(vb.x), to_tf32(vb.y), to_tf32(vb.z), to_tf32(vb.w));
    }
    fence_proxy_async_smem();
    if (warp == 0) tmem_alloc(&s_tmem, 128);
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = s_tmem;
    if (tid == 0) {
        const uint32_t sbo = (uint32_t)(k / 4) * 128u;
        const uint32_t idesc = idesc_tf32(kGramRows, kGramRows);
        for (int s = 0; s < k / 8; ++s) {
            const uint64_t ad = smem_desc(smem_u32(As) + 256u * s, 128u, sbo);
            const uint64_t bd = smem_desc(smem_u32(Bs) + 256u * s, 128u, sbo);
            mma_tf32(tmem, ad, bd, idesc, s > 0 ? 1u : 0u);
        }
        mma_commit(&s_bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&s_bar, 0);
    if (!ok && lane == 0) atomicExch(&flags[kFlagRefineTimeout], 1);
    tc_fence_after_sync();
    if (ok) {
        for (int cb = 0; cb < kGramRows / 32; ++cb) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32u * cb, v);
            tmem_ld_wait();
            float *row = out + (int64_t)(32 * warp + lane) * kGramRows + 32 * cb;
#pragma unroll
            for (int j = 0; j < 32; ++j) row[j] = __uint_as_float(v[j]);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

cudaError_t gram_tf32(const float *a, const float *b, int k, float *out, int *flags, cudaStream_t s,
                      int64_t *launches)
{
    const size_t smem = (size_t)2 * kGramRows * k * 4;
    HISS_TRY(cudaFuncSetAttribute(k_gram_tf32, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    k_gram_tf32<<<1, 128, smem, s>>>(a, b, k, out, flags);
    ++*launches;
    return cudaGetLastError();
}

}  // namespace hiss
