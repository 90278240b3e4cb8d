// noalloc.cu -- gemm_tf32_noalloc: gemm_tf32_ws for callers that cannot
// hand over a workspace because they cannot allocate device memory at all.
// Examples: code running inside a host framework whose memory pool owns all
// of the device's memory and refuses side allocations; latency-critical
// loops where an allocation, which may synchronise the device, is not
// acceptable.
//
// The scratch is a fixed, file-scope device array: every GPU that loads this
// library holds it (kNoAllocScratchBytes) until the process exits, whether
// or not the entry point is used.  Host code cannot use the array's name as
// a device address (on the host it only stands for the symbol), so the
// entry point looks the address up with cudaGetSymbolAddress, once per
// device, with that device current, and passes the pointer on.
//
// All calls share the one array.  Each call rewrites every byte of it that
// it later reads (the repacked operands, including their zero padding), so
// nothing has to start at zero and nothing left by a previous call is used.
// Two calls whose work overlaps on the GPU -- on different streams, or on
// the same device from different host threads without ordering -- race on
// the array and may corrupt each other's results.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dgemm.h"

namespace {

constexpr int64_t kNoAllocScratchBytes = DGEMM_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The device address of g_noalloc_scratch on the current device, looked up
// on the first call made with that device current (nullptr if the lookup
// failed).  A failed lookup leaves its error in the runtime's error state for
// the caller to read with cudaPeekAtLastError / cudaGetLastError; nothing
// here clears that state, so no error the caller had pending is swallowed.
void *scratch_address()
{
    static void *addr[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(once[dev], [dev] {
        void *p = nullptr;
        addr[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess ? p : nullptr;
    });
    return addr[dev];
}

}  // namespace

extern "C" int gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                 int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                 int64_t ldc, cudaStream_t stream)
{
    const int64_t need = gemm_tf32_workspace_bytes(M, N, K, A, lda, B, ldb);
    if (need < 0 || need > kNoAllocScratchBytes) return DGEMM_ERR_INVALID_ARG;
    if (need == 0 || M == 0 || N == 0 || K == 0 || alpha == 0.f)
        return gemm_tf32_ws(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr, 0, stream);
    void *scratch = scratch_address();
    if (!scratch) return DGEMM_ERR_LAUNCH;
    return gemm_tf32_ws(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, scratch, kNoAllocScratchBytes, stream);
}
