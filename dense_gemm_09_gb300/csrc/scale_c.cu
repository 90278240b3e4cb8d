// scale_c.cu -- C = beta * C for the K == 0 / alpha == 0 cases, where the
// product term is absent and A, B are not read (beta == 0 writes zeros and
// never reads C).  Memory-bound: one pass over C, grid-stride over rows,
// coalesced along each row.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

#define DGEMM_UNIT 4
#include "checked.cuh"

namespace dgemm {
namespace {

constexpr int kThreads = 256;

__global__ void scale_f32_kernel(int64_t M, int64_t N, float beta, float *__restrict__ C,
                                 int64_t ldc)
{
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        float *row = C + m * ldc;
        for (int64_t n = threadIdx.x; n < N; n += blockDim.x)
            if (DGEMM_CHECK(n < ldc)) row[n] = (beta == 0.f) ? 0.f : beta * row[n];
    }
}

__global__ void scale_f16_kernel(int64_t M, int64_t N, float beta, __half *__restrict__ C,
                                 int64_t ldc)
{
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        __half *row = C + m * ldc;
        for (int64_t n = threadIdx.x; n < N; n += blockDim.x)
            if (DGEMM_CHECK(n < ldc)) row[n] = (beta == 0.f) ? __float2half_rn(0.f)
                                   : __float2half_rn(beta * __half2float(row[n]));
    }
}

__global__ void scale_bf16_kernel(int64_t M, int64_t N, float beta, __nv_bfloat16 *__restrict__ C,
                                  int64_t ldc)
{
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        __nv_bfloat16 *row = C + m * ldc;
        for (int64_t n = threadIdx.x; n < N; n += blockDim.x)
            if (DGEMM_CHECK(n < ldc)) row[n] = (beta == 0.f) ? __float2bfloat16_rn(0.f)
                                   : __float2bfloat16_rn(beta * __bfloat162float(row[n]));
    }
}

unsigned grid_for(int64_t M)
{
    return static_cast<unsigned>(M < 65536 ? M : 65536);
}

}  // namespace

const char *launch_scale_f32(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                             cudaStream_t stream)
{
    scale_f32_kernel<<<grid_for(M), kThreads, 0, stream>>>(M, N, beta, C, ldc);
    return "scale_c_f32";
}

const char *launch_scale_f16(int64_t M, int64_t N, float beta, uint16_t *C, int64_t ldc,
                             cudaStream_t stream)
{
    scale_f16_kernel<<<grid_for(M), kThreads, 0, stream>>>(M, N, beta,
                                                           reinterpret_cast<__half *>(C), ldc);
    return "scale_c_f16";
}

const char *launch_scale_bf16(int64_t M, int64_t N, float beta, uint16_t *C, int64_t ldc,
                              cudaStream_t stream)
{
    scale_bf16_kernel<<<grid_for(M), kThreads, 0, stream>>>(M, N, beta,
                                                            reinterpret_cast<__nv_bfloat16 *>(C), ldc);
    return "scale_c_bf16";
}

}  // namespace dgemm

DGEMM_DEFINE_CHECK_READER(check_status_scale)
