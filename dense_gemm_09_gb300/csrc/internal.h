// internal.h -- declarations shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace dgemm {

inline bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Each launcher enqueues its kernel(s) on `stream` and returns the name of
// the variant it chose.  Arguments have been validated by the caller.


// C = beta * C (beta == 0: C = 0), for K == 0 or alpha == 0.
const char *launch_scale_f32(int64_t M, int64_t N, float beta, float *C, int64_t ldc,
                             cudaStream_t stream);
const char *launch_scale_f16(int64_t M, int64_t N, float beta, uint16_t *C, int64_t ldc,
                             cudaStream_t stream);
const char *launch_scale_bf16(int64_t M, int64_t N, float beta, uint16_t *C, int64_t ldc,
                              cudaStream_t stream);

struct DeviceInfo {
    int major = 0, minor = 0;
    int sm_count = 0;
    int max_smem_optin = 0;
};

// FP32 SIMT path: the one-tile-per-CTA kernel, plus a split-K launch in
// clusters for the last partial wave (or for the whole of a small problem).
const char *launch_sgemm_simt(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                              int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                              int64_t ldc, cudaStream_t stream, const DeviceInfo &dev);

// Whether the FP32 SIMT path would run this problem as one plain launch (at
// least a wave of tiles, or K too short to split) -- the case in which
// TMA-describable operands take the TMA-fed kernel.
bool sgemm_simt_plain_launch(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev);

// FP32 SIMT path fed by TMA (A and B with 16-byte aligned bases and row
// pitches; the caller checks that).  nullptr if it cannot be used for this
// call (sizes beyond TMA's coordinates, a refused tensor map), in which case
// nothing was launched.
const char *launch_sgemm_tma(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float beta, float *C, int64_t ldc, cudaStream_t stream);

// Device status word of the TMA-fed SIMT kernel (see dgemm_device_status).
int simt_read_status(int clear);

// A 2-D tiled tensor map with zero fill out of range (false if the driver's
// encoder is unavailable or refuses the description).
bool encode_tiled_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// The stall requested by dgemm_test_inject_stall for the next launch of a
// kernel with bounded waits on this host thread (its wait limit in ns, 0 if
// none); taking it clears the request.
uint64_t take_injected_stall();

// Each unit's checked-build words (checked.cuh): status 0 or
// DGEMM_ERR_BOUNDS, *site the first failed check; reset when clear != 0.
// Always 0 in the normal build.
int check_status_simt(int clear, int *site);
int check_status_tma(int clear, int *site);
int check_status_umma(int clear, int *site);
int check_status_scale(int clear, int *site);
int check_status_repack(int clear, int *site);

// Rows taken off M for the C-store checks of the next TMA-fed SIMT launch
// on this host thread (dgemm_test_shrink_bounds); taking it clears it.
int64_t take_shrink_bounds();

// Tensor-core paths: operand kinds (TN = B stored N x K, NN = B stored K x N).
enum UmmaKind { kUmmaF16TN = 0, kUmmaTF32NN = 1, kUmmaBF16TN = 2, kUmmaF16NN = 3, kUmmaBF16NN = 4 };

// Returns nullptr if the launch could not be prepared (e.g. the driver's
// tensor-map encoder is unavailable).  n_b >= N is the number of columns of
// B the kernels may read (N-major B only; columns N..n_b-1 must be zeros),
// which lets a padded copy of B take whole 128-byte column groups.
const char *launch_umma(int kind, int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                        int64_t lda, const void *B, int64_t ldb, float beta, void *C, int64_t ldc,
                        cudaStream_t stream, const DeviceInfo &dev, int64_t n_b = 0);

// Copy a rows x cols FP32 matrix (row pitch ld_src, any 4-byte alignment)
// into dst (16-byte aligned, row pitch ld_dst a multiple of 4), writing zeros
// in columns cols..ld_dst-1; false if the launch failed.
bool launch_repack_f32(const float *src, int64_t rows, int64_t cols, int64_t ld_src, float *dst,
                       int64_t ld_dst, cudaStream_t stream, const DeviceInfo &dev);

// Device status word of the tensor-core kernels (see dgemm_device_status).
int umma_read_status(int clear);

// Test hook behind dgemm_test_inject_stall.
void umma_inject_stall(uint64_t wait_limit_ns);

// Tuning hook behind dgemm_tune_next.
int umma_tune_next(int variant, int bn, int split);

// Test hooks behind dgemm_test_pair_units, dgemm_test_stream_k_tiles and
// dgemm_test_choose_config (host computation only).
int64_t umma_test_pair_units(int64_t tiles, int64_t pairs, int64_t num_kb, int64_t sk_tiles, int64_t pair,
                             int64_t *out, int64_t max_units);
int64_t umma_test_stream_k_tiles(int64_t tiles, int64_t pairs, int64_t num_kb, int wide, int mode);
int umma_test_choose(int kind, int64_t M, int64_t N, int64_t K, int sm_count, int *variant, int *bn, int *split);

}  // namespace dgemm
