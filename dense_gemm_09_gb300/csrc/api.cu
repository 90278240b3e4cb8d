// api.cu -- the C ABI declared in include/dgemm.h: argument validation on
// the host, the device check, the special cases (M or N empty; K == 0 or
// alpha == 0) and dispatch to the kernels.  Nothing here allocates device
// memory or synchronises (except dgemm_device_status, which says so).
//
// The pages' host launchers ("SGEMM CUDA代码学习", its torch bindings) check
// dtype and shape and throw; here every check returns a status before any
// launch, and launch errors are reported instead of ignored.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dgemm.h"
#include "internal.h"

namespace dgemm {
namespace {

constexpr int kMaxDevices = 64;

thread_local const char *t_last_kernel = "";

// Per-device properties, filled on first use.
bool device_info(DeviceInfo &out)
{
    static DeviceInfo cache[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    static bool valid[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::call_once(once[dev], [dev] {
        DeviceInfo d;
        bool ok = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                  cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
                      cudaSuccess;
        cache[dev] = d;
        valid[dev] = ok;
    });
    out = cache[dev];
    return valid[dev];
}

int check_device(DeviceInfo &dev)
{
    if (!device_info(dev)) return DGEMM_ERR_UNSUPPORTED_DEVICE;
    if (dev.major != 10 || dev.minor != 3) return DGEMM_ERR_UNSUPPORTED_DEVICE;
    return DGEMM_OK;
}

// Validation common to all entry points.  b_row_len is the length of a
// stored row of B (N for NN, K for TN).
int validate(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
             const void *B, int64_t ldb, int64_t b_row_len, const void *C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return DGEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < b_row_len || ldc < N) return DGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DGEMM_OK;
    if (!C) return DGEMM_ERR_INVALID_ARG;
    const bool reads_ab = K > 0 && alpha != 0.f;
    if (reads_ab && (!A || !B)) return DGEMM_ERR_INVALID_ARG;
    return DGEMM_OK;
}

// The checked build's bounds-check words of every unit, combined: the first
// nonzero status, and the site of that unit's first failed check.
int checks_failed(int clear, int *site)
{
    int (*const readers[])(int, int *) = {check_status_simt, check_status_tma, check_status_umma,
                                          check_status_scale, check_status_repack};
    int status = DGEMM_OK, where = 0;
    for (auto rd : readers) {
        int s = 0;
        const int st = rd(clear, &s);
        if (st != DGEMM_OK && status == DGEMM_OK) {
            status = st;
            where = s;
        }
    }
    if (site) *site = where;
    return status;
}

thread_local int64_t t_shrink_rows = 0;

int finish(const char *name)
{
    if (!name) return DGEMM_ERR_LAUNCH;
    const cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return DGEMM_ERR_LAUNCH;
    t_last_kernel = name;
    return DGEMM_OK;
}

}  // namespace
}  // namespace dgemm

using namespace dgemm;

extern "C" int gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                        cudaStream_t stream)
{
    int st = validate(M, N, K, alpha, A, lda, B, ldb, N, C, ldc);
    if (st != DGEMM_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = check_device(dev)) != DGEMM_OK) return st;
    if (K == 0 || alpha == 0.f) return finish(launch_scale_f32(M, N, beta, C, ldc, stream));
    return finish(launch_sgemm_simt(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev));
}

extern "C" int gemm_tf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                         const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                         cudaStream_t stream)
{
    int st = validate(M, N, K, alpha, A, lda, B, ldb, N, C, ldc);
    if (st != DGEMM_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = check_device(dev)) != DGEMM_OK) return st;
    if (K == 0 || alpha == 0.f) return finish(launch_scale_f32(M, N, beta, C, ldc, stream));
    return finish(launch_umma(kUmmaTF32NN, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev));
}

namespace {

// Where gemm_tf32_ws puts the repacked operands.  An operand is repacked
// when TMA cannot describe it (base or row pitch not a multiple of 16 bytes):
// A becomes M x round_up(K, 4) at offset 0, B K x round_up(N, 32) at a
// 256-byte boundary after it (columns past N are zeros).  bytes = 0 when neither needs it; -1 if the
// sizes overflow.
struct Tf32Repack {
    bool a = false, b = false;
    int64_t lda = 0, ldb = 0;
    int64_t off_b = 0, bytes = 0;
};

bool tma_ok_f32(const void *p, int64_t ld)
{
    return aligned16(p) && (ld * 4) % 16 == 0;
}

Tf32Repack plan_tf32_repack(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                            const float *B, int64_t ldb)
{
    Tf32Repack r;
    if (M <= 0 || N <= 0 || K <= 0) return r;
    r.a = !tma_ok_f32(A, lda);
    r.b = !tma_ok_f32(B, ldb);
    r.lda = (K + 3) / 4 * 4;
    // B padded to whole 32-column groups (zeros): the TF32 kernels then load
    // a stage's B half as one 3-D box
    r.ldb = (N + 31) / 32 * 32;
    constexpr int64_t kMax = INT64_MAX / 8;
    int64_t size_a = 0, size_b = 0;
    if (r.a) {
        if (M > kMax / r.lda) return Tf32Repack{false, false, 0, 0, 0, -1};
        size_a = (M * r.lda * 4 + 255) / 256 * 256;
    }
    if (r.b) {
        if (K > kMax / r.ldb) return Tf32Repack{false, false, 0, 0, 0, -1};
        size_b = K * r.ldb * 4;
    }
    if (size_a > kMax - size_b) return Tf32Repack{false, false, 0, 0, 0, -1};
    r.off_b = size_a;
    r.bytes = size_a + size_b;
    return r;
}

// The 16-bit entry points: kind selects the input / output type and the
// layout of B (TN: stored N x K, ldb >= K; NN: stored K x N, ldb >= N).
int gemm_16bit(int kind, bool bf16, bool nn, int64_t M, int64_t N, int64_t K, float alpha,
               const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, float beta,
               uint16_t *C, int64_t ldc, cudaStream_t stream)
{
    int st = validate(M, N, K, alpha, A, lda, B, ldb, nn ? N : K, C, ldc);
    if (st != DGEMM_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = check_device(dev)) != DGEMM_OK) return st;
    if (K == 0 || alpha == 0.f)
        return finish(bf16 ? launch_scale_bf16(M, N, beta, C, ldc, stream)
                           : launch_scale_f16(M, N, beta, C, ldc, stream));
    return finish(launch_umma(kind, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev));
}

}  // namespace

extern "C" int gemm_f16_tn(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                           int64_t lda, const uint16_t *B, int64_t ldb, float beta, uint16_t *C,
                           int64_t ldc, cudaStream_t stream)
{
    return gemm_16bit(kUmmaF16TN, false, false, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int gemm_f16_nn(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                           int64_t lda, const uint16_t *B, int64_t ldb, float beta, uint16_t *C,
                           int64_t ldc, cudaStream_t stream)
{
    return gemm_16bit(kUmmaF16NN, false, true, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int gemm_bf16_tn(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                            int64_t lda, const uint16_t *B, int64_t ldb, float beta, uint16_t *C,
                            int64_t ldc, cudaStream_t stream)
{
    return gemm_16bit(kUmmaBF16TN, true, false, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int gemm_bf16_nn(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                            int64_t lda, const uint16_t *B, int64_t ldb, float beta, uint16_t *C,
                            int64_t ldc, cudaStream_t stream)
{
    return gemm_16bit(kUmmaBF16NN, true, true, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream);
}

extern "C" int64_t gemm_tf32_workspace_bytes(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                             const float *B, int64_t ldb)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N) return -1;
    return plan_tf32_repack(M, N, K, A, lda, B, ldb).bytes;
}

extern "C" int gemm_tf32_ws(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                            const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                            void *workspace, int64_t workspace_bytes, cudaStream_t stream)
{
    int st = validate(M, N, K, alpha, A, lda, B, ldb, N, C, ldc);
    if (st != DGEMM_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = check_device(dev)) != DGEMM_OK) return st;
    if (K == 0 || alpha == 0.f) return finish(launch_scale_f32(M, N, beta, C, ldc, stream));
    const Tf32Repack r = plan_tf32_repack(M, N, K, A, lda, B, ldb);
    if (r.bytes < 0) return DGEMM_ERR_INVALID_ARG;
    if (r.bytes > 0) {
        if (!workspace || workspace_bytes < r.bytes || !aligned16(workspace)) return DGEMM_ERR_INVALID_ARG;
        float *wa = static_cast<float *>(workspace);
        float *wb = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + r.off_b);
        if (r.a) {
            if (!launch_repack_f32(A, M, K, lda, wa, r.lda, stream, dev)) return DGEMM_ERR_LAUNCH;
            A = wa;
            lda = r.lda;
        }
        if (r.b) {
            if (!launch_repack_f32(B, K, N, ldb, wb, r.ldb, stream, dev)) return DGEMM_ERR_LAUNCH;
            B = wb;
            ldb = r.ldb;
        }
    }
    return finish(launch_umma(kUmmaTF32NN, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev,
                              r.b ? r.ldb : N));
}

extern "C" int gemm_f32_ws(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                           const float *B, int64_t ldb, float beta, float *C, int64_t ldc, void *workspace,
                           int64_t workspace_bytes, cudaStream_t stream)
{
    int st = validate(M, N, K, alpha, A, lda, B, ldb, N, C, ldc);
    if (st != DGEMM_OK || M == 0 || N == 0) return st;
    DeviceInfo dev;
    if ((st = check_device(dev)) != DGEMM_OK) return st;
    if (K == 0 || alpha == 0.f) return finish(launch_scale_f32(M, N, beta, C, ldc, stream));
    // B is copied when its rows rule out 16-byte loads.  A is copied too when
    // the problem runs as one plain launch (at least a wave of tiles): with
    // both operands TMA-describable the TMA-fed kernel runs, and the copy
    // (one pass over A at HBM speed) is small against the GEMM.  Smaller
    // problems (split-K) load A element by element, so A stays in place.
    const Tf32Repack r = plan_tf32_repack(M, N, K, A, lda, B, ldb);
    if (r.bytes < 0) return DGEMM_ERR_INVALID_ARG;
    const bool copy_a = r.a && sgemm_simt_plain_launch(M, N, K, dev);
    if (r.b || copy_a) {
        if (!workspace || workspace_bytes < r.bytes || !aligned16(workspace)) return DGEMM_ERR_INVALID_ARG;
        if (copy_a) {
            float *wa = static_cast<float *>(workspace);
            if (!launch_repack_f32(A, M, K, lda, wa, r.lda, stream, dev)) return DGEMM_ERR_LAUNCH;
            A = wa;
            lda = r.lda;
        }
        if (r.b) {
            float *wb = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + r.off_b);
            if (!launch_repack_f32(B, K, N, ldb, wb, r.ldb, stream, dev)) return DGEMM_ERR_LAUNCH;
            B = wb;
            ldb = r.ldb;
        }
    }
    return finish(launch_sgemm_simt(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev));
}

extern "C" const char *dgemm_status_string(int status)
{
    switch (status) {
    case DGEMM_OK: return "DGEMM_OK: success";
    case DGEMM_ERR_INVALID_ARG: return "DGEMM_ERR_INVALID_ARG: invalid size, leading dimension or pointer";
    case DGEMM_ERR_UNSUPPORTED_DEVICE: return "DGEMM_ERR_UNSUPPORTED_DEVICE: current device is not sm_103 (GB300)";
    case DGEMM_ERR_LAUNCH: return "DGEMM_ERR_LAUNCH: the CUDA runtime reported a launch error";
    case DGEMM_ERR_TIMEOUT: return "DGEMM_ERR_TIMEOUT: a kernel wait ran out and the kernel exited early";
    case DGEMM_ERR_BOUNDS: return "DGEMM_ERR_BOUNDS: a device-side bounds check failed (checked build)";
    default: return "unknown dgemm status";
    }
}

extern "C" int dgemm_device_status(int clear)
{
    DeviceInfo dev;
    int st = check_device(dev);
    if (st != DGEMM_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return DGEMM_ERR_LAUNCH;
    const int a = umma_read_status(clear);
    const int b = simt_read_status(clear);
    if (a != DGEMM_OK) return a;
    if (b != DGEMM_OK) return b;
    return checks_failed(clear, nullptr);
}

extern "C" int dgemm_check_site(void)
{
    DeviceInfo dev;
    if (check_device(dev) != DGEMM_OK) return 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return 0;
    int site = 0;
    checks_failed(0, &site);
    return site;
}

extern "C" int dgemm_test_shrink_bounds(int64_t rows)
{
    if (rows < 0) return DGEMM_ERR_INVALID_ARG;
    t_shrink_rows = rows;
    return DGEMM_OK;
}

int64_t dgemm::take_shrink_bounds()
{
    const int64_t v = t_shrink_rows;
    t_shrink_rows = 0;
    return v;
}

extern "C" int dgemm_tune_next(int variant, int bn, int split)
{
    return umma_tune_next(variant, bn, split);
}

extern "C" int64_t dgemm_test_pair_units(int64_t tiles, int64_t pairs, int64_t num_kb, int64_t sk_tiles,
                                         int64_t pair, int64_t *out, int64_t max_units)
{
    return umma_test_pair_units(tiles, pairs, num_kb, sk_tiles, pair, out, max_units);
}

extern "C" int64_t dgemm_test_stream_k_tiles(int64_t tiles, int64_t pairs, int64_t num_kb, int wide, int mode)
{
    return umma_test_stream_k_tiles(tiles, pairs, num_kb, wide, mode);
}

extern "C" int dgemm_test_choose_config(int kind, int64_t M, int64_t N, int64_t K, int sm_count, int *variant,
                                        int *bn, int *split)
{
    return umma_test_choose(kind, M, N, K, sm_count, variant, bn, split);
}

extern "C" int dgemm_test_inject_stall(uint64_t wait_limit_ns)
{
    umma_inject_stall(wait_limit_ns);
    return DGEMM_OK;
}

extern "C" const char *dgemm_last_kernel(void)
{
    return t_last_kernel;
}
