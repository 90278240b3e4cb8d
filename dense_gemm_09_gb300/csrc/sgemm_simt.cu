// sgemm_simt.cu -- FP32 SGEMM on the CUDA cores for sm_103a:
//     C = alpha * A * B + beta * C, all row-major, FP32 fused multiply-add.
//
// Design (what is kept from the pages, and what changed for GB300):
//   * Block tile 128 x 128, K slice 16, 256 threads, 8 x 8 outputs per thread
//     held in registers -- the thread-tile idea of "SGEMM CUDA代码学习",
//     "第 2 步" and of "CUDA GEMM：从基础写法到工程优化", "5. 2D Block Tiling".
//   * A is staged transposed in shared memory (As[k][m]) and each thread's 8
//     rows are split into two groups of 4 at m and m + 64, so every shared
//     read is a conflict-free 16-byte load -- "SGEMM CUDA代码学习", "第 3 步".
//     A 4-float pad on As rows, plus a warp-to-tile mapping in which each warp
//     stores 16 rows x 2 k-quads, keeps the transposing stores conflict-free.
//   * Threads are grouped so that a warp covers a 32 x 64 piece of the tile
//     (warp tiling, "CUDA GEMM：从基础写法到工程优化", "10. Warp Tiling"):
//     each 16-byte shared read then touches 64 or 128 distinct bytes, one
//     shared-memory wavefront.
//   * Double buffering through registers: the global loads of slice k+1 are
//     issued before the FMAs of slice k and stored after them, one barrier
//     per slice -- "SGEMM CUDA代码学习", "第 4 步".
//   * Unlike the pages' kernels, every load is predicated: M, N and K tails
//     read zeros and stores are masked, and no thread leaves before a
//     barrier.  Operands whose pointers or leading dimensions are not 16-byte
//     aligned take a scalar-load instantiation.
//   * Epilogue: alpha * acc + beta * C_old, with C not read when beta == 0,
//     16-byte stores where aligned.
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace dgemm {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int THREADS = 256;
constexpr int AS_LD = BM + 4;  // padded row of the transposed A slice
constexpr int kGroupM = 8;     // rasterisation group height, in tiles

struct SimtSmem {
    float As[2][BK][AS_LD];
    float Bs[2][BK][BN];
};

// Global -> register staging of one K slice (2 float4 of A, 2 float4 of B per
// thread).  Out-of-range elements read as zero.
template <bool kVec>
struct SliceRegs {
    float4 a[2];
    float4 b[2];
};

template <bool kVec>
__device__ __forceinline__ void load_slice(SliceRegs<kVec> &r, const float *__restrict__ A,
                                           int64_t lda, const float *__restrict__ B, int64_t ldb,
                                           int64_t M, int64_t N, int64_t K, int64_t m0,
                                           int64_t n0, int64_t k0, int warp, int lane, int tid)
{
    // A: thread covers row m = warp*16 + (lane & 15), k-quads 2i + (lane >> 4).
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int m = warp * 16 + (lane & 15);
        const int kq = (i * 2 + (lane >> 4)) * 4;
        const int64_t gm = m0 + m, gk = k0 + kq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (gm < M) {
            const float *p = A + gm * lda + gk;
            if (kVec && gk + 3 < K) {
                v = __ldg(reinterpret_cast<const float4 *>(p));
            } else {
                if (gk + 0 < K) v.x = __ldg(p + 0);
                if (gk + 1 < K) v.y = __ldg(p + 1);
                if (gk + 2 < K) v.z = __ldg(p + 2);
                if (gk + 3 < K) v.w = __ldg(p + 3);
            }
        }
        r.a[i] = v;
    }
    // B: a warp reads one full 128-float row of the slice.
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = tid + i * THREADS;
        const int k = idx >> 5;
        const int nq = (idx & 31) * 4;
        const int64_t gk = k0 + k, gn = n0 + nq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (gk < K) {
            const float *p = B + gk * ldb + gn;
            if (kVec && gn + 3 < N) {
                v = __ldg(reinterpret_cast<const float4 *>(p));
            } else {
                if (gn + 0 < N) v.x = __ldg(p + 0);
                if (gn + 1 < N) v.y = __ldg(p + 1);
                if (gn + 2 < N) v.z = __ldg(p + 2);
                if (gn + 3 < N) v.w = __ldg(p + 3);
            }
        }
        r.b[i] = v;
    }
}

template <bool kVec>
__device__ __forceinline__ void store_slice(const SliceRegs<kVec> &r, SimtSmem &s, int buf,
                                            int warp, int lane, int tid)
{
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int m = warp * 16 + (lane & 15);
        const int kq = (i * 2 + (lane >> 4)) * 4;
        s.As[buf][kq + 0][m] = r.a[i].x;
        s.As[buf][kq + 1][m] = r.a[i].y;
        s.As[buf][kq + 2][m] = r.a[i].z;
        s.As[buf][kq + 3][m] = r.a[i].w;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = tid + i * THREADS;
        const int k = idx >> 5;
        const int nq = (idx & 31) * 4;
        *reinterpret_cast<float4 *>(&s.Bs[buf][k][nq]) = r.b[i];
    }
}

__device__ __forceinline__ void epilogue_store(float *__restrict__ C, int64_t ldc, int64_t M,
                                               int64_t N, int64_t gm, int64_t gn, const float *acc,
                                               float alpha, float beta, bool vec_c)
{
    if (gm >= M) return;
    float *p = C + gm * ldc + gn;
    if (vec_c && gn + 3 < N) {
        float4 o;
        o.x = alpha * acc[0];
        o.y = alpha * acc[1];
        o.z = alpha * acc[2];
        o.w = alpha * acc[3];
        if (beta != 0.f) {
            const float4 c = *reinterpret_cast<const float4 *>(p);
            o.x = fmaf(beta, c.x, o.x);
            o.y = fmaf(beta, c.y, o.y);
            o.z = fmaf(beta, c.z, o.z);
            o.w = fmaf(beta, c.w, o.w);
        }
        *reinterpret_cast<float4 *>(p) = o;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (gn + j < N) {
                float o = alpha * acc[j];
                if (beta != 0.f) o = fmaf(beta, p[j], o);
                p[j] = o;
            }
        }
    }
}

template <bool kVec>
__global__ void __launch_bounds__(THREADS, 2)
    sgemm_simt_kernel(int64_t M, int64_t N, int64_t K, float alpha, const float *__restrict__ A,
                      int64_t lda, const float *__restrict__ B, int64_t ldb, float beta,
                      float *__restrict__ C, int64_t ldc, bool vec_c)
{
    __shared__ __align__(16) SimtSmem s;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // warp tiling: 8 warps as 4 (m) x 2 (n); lanes as 4 (m) x 8 (n)
    const int ty = (warp >> 1) * 4 + (lane >> 3);  // 0..15
    const int tx = (warp & 1) * 8 + (lane & 7);    // 0..15

    // Grouped rasterisation of a 1-D grid: runs of kGroupM consecutive
    // blocks walk down M inside one N column, so blocks resident together
    // share B columns and a short band of A rows in L2.
    int64_t m_tile, n_tile;
    {
        const int64_t tiles_m = (M + BM - 1) / BM;
        const int64_t b = blockIdx.x;
        const int64_t per_group = static_cast<int64_t>(kGroupM) * ((N + BN - 1) / BN);
        const int64_t g = b / per_group, r = b % per_group;
        const int64_t gm = tiles_m - g * kGroupM < kGroupM ? tiles_m - g * kGroupM : kGroupM;
        m_tile = g * kGroupM + r % gm;
        n_tile = r / gm;
    }
    const int64_t m0 = m_tile * BM;
    const int64_t n0 = n_tile * BN;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int64_t kt_count = (K + BK - 1) / BK;
    SliceRegs<kVec> regs;
    load_slice<kVec>(regs, A, lda, B, ldb, M, N, K, m0, n0, 0, warp, lane, tid);
    store_slice<kVec>(regs, s, 0, warp, lane, tid);
    __syncthreads();

    for (int64_t kt = 0; kt < kt_count; ++kt) {
        const int buf = static_cast<int>(kt & 1);
        const bool more = kt + 1 < kt_count;
        if (more)
            load_slice<kVec>(regs, A, lda, B, ldb, M, N, K, m0, n0, (kt + 1) * BK, warp, lane, tid);

#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&s.As[buf][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&s.As[buf][k][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&s.Bs[buf][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&s.Bs[buf][k][tx * 4 + 64]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }

        if (more) store_slice<kVec>(regs, s, buf ^ 1, warp, lane, tid);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        epilogue_store(C, ldc, M, N, gm, n0 + tx * 4, &acc[i][0], alpha, beta, vec_c);
        epilogue_store(C, ldc, M, N, gm, n0 + 64 + tx * 4, &acc[i][4], alpha, beta, vec_c);
    }
}

}  // namespace

const char *launch_sgemm_simt(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                              int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                              int64_t ldc, cudaStream_t stream)
{
    const bool vec_ab = aligned16(A) && aligned16(B) && (lda % 4 == 0) && (ldb % 4 == 0);
    const bool vec_c = aligned16(C) && (ldc % 4 == 0);
    const int64_t blocks = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const dim3 grid(static_cast<unsigned>(blocks));
    if (vec_ab) {
        sgemm_simt_kernel<true><<<grid, THREADS, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb, beta,
                                                              C, ldc, vec_c);
        return "sgemm_simt_128x128x16_vec";
    }
    sgemm_simt_kernel<false><<<grid, THREADS, 0, stream>>>(M, N, K, alpha, A, lda, B, ldb, beta, C,
                                                           ldc, vec_c);
    return "sgemm_simt_128x128x16_scalar";
}

}  // namespace dgemm
