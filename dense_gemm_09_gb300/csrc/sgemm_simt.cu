// sgemm_simt.cu -- FP32 SGEMM on the CUDA cores for sm_103a:
//     C = alpha * A * B + beta * C, all row-major, FP32 fused multiply-add.
//
// Design (what is kept from the pages, and what changed for GB300):
//   * Block tile 128 x 128, K slices of 16, 256 threads, 8 x 8 outputs per
//     thread held in registers -- the thread-tile idea of "SGEMM CUDA代码学习",
//     "第 2 步", and "CUDA GEMM：从基础写法到工程优化", "5. 2D Block Tiling".
//   * A is staged transposed in shared memory (As[k][m]); each thread's 8 rows
//     (and 8 columns) are two groups of 4 at m and m + 64, so every shared
//     read is a conflict-free 16-byte load -- "SGEMM CUDA代码学习", "第 3 步".
//   * Warp tiling ("CUDA GEMM：从基础写法到工程优化", "10. Warp Tiling"): a warp
//     covers a 32 x 64 piece of the tile, so each 16-byte shared read touches
//     at most 128 distinct bytes (one wavefront).
//   * A 4-stage ring of K slices filled with cp.async, the multi-stage
//     asynchronous copy of "SGEMM CUDA代码学习", "第 5 步" and "CUDA GEMM：
//     从基础写法到工程优化", "12. Async Copy Double Buffering".  A is copied
//     element by element straight into its transposed place (no registers);
//     B in 16-byte pieces.  Copies past M, N or K are zero-filled, so tails
//     need no special loop, and no thread leaves before a barrier.
//   * The FMAs are Blackwell's packed two-lane form (fma.rn.f32x2): each
//     instruction updates two adjacent accumulators with two independent
//     single-precision fused multiply-adds, halving the FMA issue slots.
//     The arithmetic per output element is unchanged: one FP32 FMA per k, in
//     k order.
//   * Epilogue: alpha * acc + beta * C_old, C not read when beta == 0,
//     16-byte stores where aligned.
//   * Problems too small to fill the GPU (fewer tiles than resident CTAs, 2
//     per SM) run split-K in clusters of S CTAs that each sum one contiguous
//     range of K slices; the partial sums meet in distributed shared memory
//     and are added in rank order, so the result does not depend on timing.
//     This is the split-K that "如何优化一个 CUDA Matmul Kernel ... Worklog",
//     section "Kernel 10: Warptiling", finds the vendor library using at
//     size 256 (a matmul kernel, then a reduction); here the reduction
//     happens inside the cluster, with no extra memory and no second kernel.
//     (Splitting only the last partial wave of a large problem was measured
//     and lost: as a second launch it waits for the first launch's slowest
//     CTAs, and as one cluster launch the whole grid ran ~5 % slower.)
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

#define DGEMM_UNIT 1
#include "checked.cuh"

namespace dgemm {
namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int AS_LD = BM + 4;  // padded row of the transposed A slice
constexpr int kGroupM = 16;    // rasterisation group height, in tiles

struct SimtStage {
    float As[BK][AS_LD];
    float Bs[BK][BN];
};
constexpr int SMEM_BYTES = STAGES * static_cast<int>(sizeof(SimtStage));

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int kPending>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// Issue the copies of K slice `kt` into `stage`.
//   A: element (m, k) of the slice, m = warp*4 + lane/8 + 32*(e%4),
//      k = lane%8 + 8*(e/4), e = 0..7: a warp reads 8 consecutive k of 4 rows
//      (one 32-byte sector each) and writes 32 distinct banks.
//   B: row k = warp + 8*e, columns lane*4 .. lane*4+3, e = 0..1.
template <bool kVec>
__device__ __forceinline__ void load_slice(uint32_t stage_smem, const float *__restrict__ A,
                                           int64_t lda, const float *__restrict__ B, int64_t ldb,
                                           int64_t M, int64_t N, int64_t K, int64_t m0, int64_t n0,
                                           int64_t kt, int warp, int lane)
{
    const int64_t k0 = kt * BK;
    const uint32_t as = stage_smem;
    const uint32_t bs = stage_smem + static_cast<uint32_t>(offsetof(SimtStage, Bs));
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int m = warp * 4 + (lane >> 3) + 32 * (e & 3);
        const int k = (lane & 7) + 8 * (e >> 2);
        const int64_t gm = m0 + m, gk = k0 + k;
        const bool ok = gm < M && gk < K;
        const float *src = ok ? A + gm * lda + gk : A;
        if (DGEMM_CHECK(m < BM && k < BK))  // the transposed slot lies inside As
            cp_async4(as + static_cast<uint32_t>((k * AS_LD + m) * 4), src, ok ? 4u : 0u);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int k = warp + 8 * e;
        const int n = lane * 4;
        const int64_t gk = k0 + k, gn = n0 + n;
        const uint32_t dst = bs + static_cast<uint32_t>((k * BN + n) * 4);
        if (!DGEMM_CHECK(k < BK && n + 3 < BN)) continue;  // the four slots lie inside Bs
        if constexpr (kVec) {
            const int64_t left = gk < K ? N - gn : 0;
            const uint32_t bytes = left >= 4 ? 16u : (left > 0 ? static_cast<uint32_t>(left) * 4u : 0u);
            cp_async16(dst, bytes ? B + gk * ldb + gn : B, bytes);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = gk < K && gn + j < N;
                cp_async4(dst + 4 * j, ok ? B + gk * ldb + gn + j : B, ok ? 4u : 0u);
            }
        }
    }
}

__device__ __forceinline__ void epilogue_store(float *__restrict__ C, int64_t ldc, int64_t M,
                                               int64_t N, int64_t gm, int64_t gn, const float *acc,
                                               float alpha, float beta, bool vec_c)
{
    if (gm >= M) return;
    float *p = C + gm * ldc + gn;
    if (vec_c && gn + 3 < N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(p) & 15u) == 0)) {
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

// ---- split-K across a cluster (the last partial wave, and small problems)
//
// The S CTAs of a cluster (S in {2, 3, 4, 5, 8}) share one tile; rank r sums
// K slices [r*kt/S, (r+1)*kt/S).  Row i (0..7) of each thread's eight rows
// belongs to rank i mod S.  Every rank stores the rows it does not own into
// the owner's stage ring (idle by then) with remote 16-byte stores; after a
// cluster barrier each owner adds the S partials in rank order 0..S-1 and
// runs the ordinary epilogue on its rows.  Receive layout, in float4 units:
// [sender slot among the other S-1 ranks][row index i/S][half h][thread],
// so a warp's stores and loads are 512 contiguous bytes.
constexpr int kSplitChoices[] = {8, 5, 4, 3, 2};

__host__ __device__ constexpr uint32_t split_recv_bytes(uint32_t S)
{
    return (S - 1) * ((8 + S - 1) / S) * 2 * THREADS * 16;
}
static_assert(split_recv_bytes(2) <= uint32_t(SMEM_BYTES) && split_recv_bytes(3) <= uint32_t(SMEM_BYTES) &&
                  split_recv_bytes(4) <= uint32_t(SMEM_BYTES) && split_recv_bytes(5) <= uint32_t(SMEM_BYTES) &&
                  split_recv_bytes(8) <= uint32_t(SMEM_BYTES),
              "split-K partials must fit in the stage ring");

__device__ __forceinline__ uint32_t split_recv_offset(uint32_t slot, uint32_t il, uint32_t h,
                                                      uint32_t S, int tid)
{
    const uint32_t il_max = (8 + S - 1) / S;
    return (((slot * il_max + il) * 2 + h) * THREADS + static_cast<uint32_t>(tid)) * 16;
}

__device__ __forceinline__ void split_reduce_store(const float2 (&acc)[8][4], uint32_t smem0,
                                                   uint32_t S, uint32_t rank, int tid,
                                                   float *__restrict__ C, int64_t ldc, int64_t M,
                                                   int64_t N, int64_t m0, int64_t n0, int ty,
                                                   int tx, float alpha, float beta, bool vec_c)
{
    ptx::cluster_sync();  // every CTA of the cluster is done with its stage ring
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t owner = static_cast<uint32_t>(i) % S;
        if (owner == rank) continue;
        const uint32_t slot = rank < owner ? rank : rank - 1;
        const uint32_t off = split_recv_offset(slot, static_cast<uint32_t>(i) / S, 0, S, tid);
        // both 16-byte words land inside the owner's stage ring
        if (!DGEMM_CHECK(owner < S && off + THREADS * 16 + 16 <= static_cast<uint32_t>(SMEM_BYTES))) continue;
        const uint32_t dst = ptx::mapa(smem0 + off, owner);
        ptx::st_shared_cluster_v4(dst, make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y));
        ptx::st_shared_cluster_v4(dst + THREADS * 16,
                                  make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y));
    }
    ptx::cluster_sync();  // the partials have landed in their owners
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (static_cast<uint32_t>(i) % S != rank) continue;
        float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
        for (uint32_t q = 0; q < S; ++q) {
            float4 l, h;
            if (q == rank) {
                l = make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
                h = make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y);
            } else {
                const uint32_t slot = q < rank ? q : q - 1;
                const uint32_t off = split_recv_offset(slot, static_cast<uint32_t>(i) / S, 0, S, tid);
                if (DGEMM_CHECK(off + THREADS * 16 + 16 <= static_cast<uint32_t>(SMEM_BYTES))) {
                    l = ptx::ld_shared_v4f(smem0 + off);
                    h = ptx::ld_shared_v4f(smem0 + off + THREADS * 16);
                } else {
                    l = h = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            lo[0] += l.x; lo[1] += l.y; lo[2] += l.z; lo[3] += l.w;
            hi[0] += h.x; hi[1] += h.y; hi[2] += h.z; hi[3] += h.w;
        }
        const int64_t gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        epilogue_store(C, ldc, M, N, gm, n0 + tx * 4, lo, alpha, beta, vec_c);
        epilogue_store(C, ldc, M, N, gm, n0 + 64 + tx * 4, hi, alpha, beta, vec_c);
    }
}

// Launch modes.
//   kPlain : one CTA per tile, tile tile0 + blockIdx.x.
//   kSplit : clusters of S; cluster c splits tile tile0 + c over K.
enum SimtMode { kPlain = 0, kSplit = 1 };

// This CTA's share of its tile: S ranks split the tile's K slices (S = 1:
// the whole tile); rank is the CTA's place among them.
template <int kMode>
__device__ __forceinline__ void split_role(uint32_t &S, uint32_t &rank)
{
    S = 1;
    rank = 0;
    if constexpr (kMode == kSplit) {
        S = ptx::cluster_nctarank();
        rank = ptx::cluster_ctarank();
    }
}

template <bool kVec, int kMode>
__global__ void __launch_bounds__(THREADS, 2)
    sgemm_simt_kernel(int64_t M, int64_t N, int64_t K, float alpha, const float *__restrict__ A,
                      int64_t lda, const float *__restrict__ B, int64_t ldb, float beta,
                      float *__restrict__ C, int64_t ldc, int64_t tile0, bool vec_c)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SimtStage *stages = reinterpret_cast<SimtStage *>(smem_raw);
    const uint32_t smem0 = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    // warp tiling: 8 warps as 4 (m) x 2 (n); lanes as 4 (m) x 8 (n)
    const int ty = (warp >> 1) * 4 + (lane >> 3);  // 0..15
    const int tx = (warp & 1) * 8 + (lane & 7);    // 0..15

    // Grouped rasterisation of a 1-D grid: runs of kGroupM consecutive blocks
    // walk down M inside one N column, so blocks resident together share B
    // columns and a short band of A rows in L2.
    uint32_t S, rank;
    split_role<kMode>(S, rank);
    const int64_t b = tile0 + blockIdx.x / S;
    int64_t m0, n0;
    {
        const int64_t tiles_m = (M + BM - 1) / BM;
        const int64_t per_group = static_cast<int64_t>(kGroupM) * ((N + BN - 1) / BN);
        const int64_t g = b / per_group, r = b % per_group;
        const int64_t gm = tiles_m - g * kGroupM < kGroupM ? tiles_m - g * kGroupM : kGroupM;
        m0 = (g * kGroupM + r % gm) * BM;
        n0 = (r / gm) * BN;
    }

    float2 acc[8][4];  // acc[i][j]: row i, columns 2j and 2j+1 of the thread's 8
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);

    const int64_t kt_count = (K + BK - 1) / BK;
    // (the host splits only when kt_count < 2^28, so 32-bit products suffice)
    constexpr bool kMaySplit = kMode != kPlain;
    const int64_t kt0 = kMaySplit ? static_cast<int64_t>(rank * static_cast<uint32_t>(kt_count) / S) : 0;
    int64_t kt1 = kMaySplit ? static_cast<int64_t>((rank + 1) * static_cast<uint32_t>(kt_count) / S) : kt_count;
    // the raster maps the CTA onto a tile inside C, and the thread's fragment
    // columns (ty * 4 .. ty * 4 + 67, tx * 4 .. tx * 4 + 67) lie inside the
    // slice rows; otherwise the CTA loads and stores nothing
    if (!DGEMM_CHECK_CTA(m0 >= 0 && m0 < M && n0 >= 0 && n0 < N && ty < 16 && tx < 16)) kt1 = kt0;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (kt0 + s < kt1)
            load_slice<kVec>(smem0 + s * sizeof(SimtStage), A, lda, B, ldb, M, N, K, m0, n0, kt0 + s,
                             warp, lane);
        cp_async_commit();
    }

    int read_stage = 0, write_stage = STAGES - 1;
    for (int64_t kt = kt0; kt < kt1; ++kt) {
        cp_async_wait<STAGES - 2>();  // slice kt has landed (this thread's copies)
        __syncthreads();              // ... everyone's; and slice kt-1 is consumed
        if (kt + STAGES - 1 < kt1)
            load_slice<kVec>(smem0 + static_cast<uint32_t>(write_stage) * sizeof(SimtStage), A, lda,
                             B, ldb, M, N, K, m0, n0, kt + STAGES - 1, warp, lane);
        cp_async_commit();
        write_stage = write_stage + 1 == STAGES ? 0 : write_stage + 1;
        const SimtStage &st = stages[read_stage];
        read_stage = read_stage + 1 == STAGES ? 0 : read_stage + 1;
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&st.As[k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&st.As[k][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&st.Bs[k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&st.Bs[k][tx * 4 + 64]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                  make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 a2 = make_float2(av[i], av[i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(a2, bp[j], acc[i][j]);
            }
        }
    }
    cp_async_wait<0>();

    if constexpr (kMaySplit) {
        // S and rank are read again here rather than kept live through the loop
        split_role<kMode>(S, rank);
        split_reduce_store(acc, smem0, S, rank, tid, C, ldc, M, N, m0, n0, ty, tx, alpha, beta, vec_c);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
            const float lo[4] = {acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y};
            const float hi[4] = {acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y};
            epilogue_store(C, ldc, M, N, gm, n0 + tx * 4, lo, alpha, beta, vec_c);
            epilogue_store(C, ldc, M, N, gm, n0 + 64 + tx * 4, hi, alpha, beta, vec_c);
        }
    }
}

// Occupancy facts of one kernel variant on one device, computed once.
struct SimtOccupancy {
    bool ready = false;
    int blocks_per_sm = 0;      // resident CTAs per SM of the one-tile-per-CTA kernel
    int clusters[9] = {};       // co-resident clusters of the split kernel, by size
};

template <bool kVec>
const SimtOccupancy &occupancy(int device)
{
    constexpr int kMaxDevices = 64;
    static SimtOccupancy table[kMaxDevices];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    SimtOccupancy &o = table[device >= 0 && device < kMaxDevices ? device : 0];
    if (o.ready) return o;
    cudaFuncSetAttribute(sgemm_simt_kernel<kVec, kPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
    cudaFuncSetAttribute(sgemm_simt_kernel<kVec, kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o.blocks_per_sm, sgemm_simt_kernel<kVec, kPlain>,
                                                      THREADS, SMEM_BYTES) != cudaSuccess)
        o.blocks_per_sm = 1;
    for (int S : kSplitChoices) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(S);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(S));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sgemm_simt_kernel<kVec, kSplit>, &cfg) != cudaSuccess) n = 0;
        o.clusters[S] = n;
    }
    cudaGetLastError();  // a refused query leaves no sticky error behind
    o.ready = true;
    return o;
}

// How one call is launched.  With W resident CTAs (2 per SM): fewer tiles
// than W take one kSplit launch in clusters of the largest S in
// {8, 5, 4, 3, 2} with tiles * S <= W, at least two K slices per rank and
// every cluster resident at once; anything else one kPlain launch.
struct SimtPlan {
    int mode;
    int split;  // S (1: no split)
};

SimtPlan plan_simt(int64_t tiles, int64_t kt_count, int64_t W, const SimtOccupancy &occ)
{
    if (W > 0 && tiles < W && kt_count < (int64_t(1) << 28)) {
        for (int S : kSplitChoices)
            if (tiles * S <= W && kt_count >= 2 * S && tiles <= occ.clusters[S]) return SimtPlan{kSplit, S};
    }
    return SimtPlan{kPlain, 1};
}

template <bool kVec, int kMode>
bool launch_clusters(int S, int64_t grid, int64_t tile0, int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                     int64_t ldc, bool vec_c, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sgemm_simt_kernel<kVec, kMode>, M, N, K, alpha, A, lda, B, ldb, beta,
                              C, ldc, tile0, vec_c) == cudaSuccess;
}

template <bool kVec>
bool launch_kernel(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                   const float *B, int64_t ldb, float beta, float *C, int64_t ldc, bool vec_c,
                   cudaStream_t stream, const DeviceInfo &dev, SimtPlan &pl)
{
    int device = 0;
    cudaGetDevice(&device);
    const SimtOccupancy &occ = occupancy<kVec>(device);
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    pl = plan_simt(tiles, (K + BK - 1) / BK, static_cast<int64_t>(occ.blocks_per_sm) * dev.sm_count, occ);
    if (pl.mode == kSplit)
        return launch_clusters<kVec, kSplit>(pl.split, tiles * pl.split, 0, M, N, K, alpha, A, lda, B, ldb,
                                             beta, C, ldc, vec_c, stream);
    sgemm_simt_kernel<kVec, kPlain><<<static_cast<unsigned>(tiles), THREADS, SMEM_BYTES, stream>>>(
        M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 0, vec_c);
    return true;
}

// Variant name of the launch a plan makes.
const char *simt_name(bool vec, const SimtPlan &pl)
{
    static const char *const kPlainName[2] = {"sgemm_simt_128x128x16_ffma2_cpasync4",
                                              "sgemm_simt_128x128x16_ffma2_cpasync16"};
    static const char *const kSplitName[2][9] = {
        {nullptr, nullptr, "sgemm_simt_splitk2_128x128x16_ffma2_cpasync4",
         "sgemm_simt_splitk3_128x128x16_ffma2_cpasync4", "sgemm_simt_splitk4_128x128x16_ffma2_cpasync4",
         "sgemm_simt_splitk5_128x128x16_ffma2_cpasync4", nullptr, nullptr,
         "sgemm_simt_splitk8_128x128x16_ffma2_cpasync4"},
        {nullptr, nullptr, "sgemm_simt_splitk2_128x128x16_ffma2_cpasync16",
         "sgemm_simt_splitk3_128x128x16_ffma2_cpasync16", "sgemm_simt_splitk4_128x128x16_ffma2_cpasync16",
         "sgemm_simt_splitk5_128x128x16_ffma2_cpasync16", nullptr, nullptr,
         "sgemm_simt_splitk8_128x128x16_ffma2_cpasync16"}};
    const int v = vec ? 1 : 0;
    if (pl.mode == kSplit && pl.split >= 2 && pl.split <= 8 && kSplitName[v][pl.split])
        return kSplitName[v][pl.split];
    return kPlainName[v];
}

}  // namespace

bool sgemm_simt_plain_launch(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev)
{
    int device = 0;
    cudaGetDevice(&device);
    const SimtOccupancy &occ = occupancy<true>(device);
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    return plan_simt(tiles, (K + BK - 1) / BK, static_cast<int64_t>(occ.blocks_per_sm) * dev.sm_count, occ).mode ==
           kPlain;
}

const char *launch_sgemm_simt(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                              int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                              int64_t ldc, cudaStream_t stream, const DeviceInfo &dev)
{
    // 16-byte copies of B need a 16-byte aligned base and row pitch.
    const bool vec_b = aligned16(B) && (ldb % 4 == 0);
    const bool vec_c = aligned16(C) && (ldc % 4 == 0);
    // Problems of at least a wave of tiles whose A and B TMA can describe
    // take the TMA-fed kernel (sgemm_tma.cu).
    if (vec_b && aligned16(A) && (lda % 4 == 0) && sgemm_simt_plain_launch(M, N, K, dev)) {
        if (const char *name = launch_sgemm_tma(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))
            return name;
    }
    SimtPlan pl{kPlain, 1};
    const bool ok =
        vec_b ? launch_kernel<true>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, vec_c, stream, dev, pl)
              : launch_kernel<false>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, vec_c, stream, dev, pl);
    // a refused cluster launch is reported through the runtime's error state,
    // which the caller reads; the name still says what was attempted
    (void)ok;
    return simt_name(vec_b, pl);
}

}  // namespace dgemm

DGEMM_DEFINE_CHECK_READER(check_status_simt)
