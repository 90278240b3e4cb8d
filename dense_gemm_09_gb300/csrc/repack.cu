// repack.cu -- copies a row-major FP32 operand whose base or row pitch TMA
// cannot describe (not a 16-byte multiple) into a caller-provided buffer
// with a 16-byte-aligned base and pitch, so that the tensor-core kernels can
// load it with TMA.  Used by gemm_tf32_ws; the values are copied bit for bit.
//
// The copy is bound by HBM bandwidth: each block takes whole rows, its
// threads walk a row in 16-byte chunks (four 4-byte loads -- the source row
// is only 4-byte aligned -- and one 16-byte store).  Columns past the last
// one of a row up to the padded pitch are written as zeros (the caller may
// let the GEMM read them as extra zero columns).
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

#define DGEMM_UNIT 5
#include "checked.cuh"

namespace dgemm {
namespace {

constexpr int kRepackThreads = 256;
constexpr int kRepackBlocksPerSm = 8;

__global__ void __launch_bounds__(kRepackThreads)
    repack_rows_f32(const float *__restrict__ src, int64_t rows, int64_t cols, int64_t ld_src,
                    float *__restrict__ dst, int64_t ld_dst)
{
    const int64_t chunks = ld_dst / 4;  // the whole padded row
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float *s = src + r * ld_src;
        float4 *d = reinterpret_cast<float4 *>(dst + r * ld_dst);
        for (int64_t q = threadIdx.x; q < chunks; q += blockDim.x) {
            const int64_t c = q * 4;
            float4 v;
            v.x = c < cols ? s[c] : 0.f;
            v.y = c + 1 < cols ? s[c + 1] : 0.f;
            v.z = c + 2 < cols ? s[c + 2] : 0.f;
            v.w = c + 3 < cols ? s[c + 3] : 0.f;
            // the 16-byte store is aligned and stays inside the padded row
            if (DGEMM_CHECK(c + 3 < ld_dst && (reinterpret_cast<uintptr_t>(d + q) & 15u) == 0)) d[q] = v;
        }
    }
}

}  // namespace

bool launch_repack_f32(const float *src, int64_t rows, int64_t cols, int64_t ld_src, float *dst,
                       int64_t ld_dst, cudaStream_t stream, const DeviceInfo &dev)
{
    if (rows <= 0 || cols <= 0) return true;
    const int64_t cap = static_cast<int64_t>(dev.sm_count > 0 ? dev.sm_count : 1) * kRepackBlocksPerSm;
    const int64_t grid = rows < cap ? rows : cap;
    repack_rows_f32<<<static_cast<unsigned>(grid), kRepackThreads, 0, stream>>>(src, rows, cols, ld_src, dst,
                                                                                 ld_dst);
    return cudaPeekAtLastError() == cudaSuccess;
}

}  // namespace dgemm

DGEMM_DEFINE_CHECK_READER(check_status_repack)
