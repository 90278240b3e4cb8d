// sgemm_tma.cu -- FP32 SGEMM on the CUDA cores for sm_103a, operands staged
// by TMA:  C = alpha * A * B + beta * C, all row-major, FP32 fused
// multiply-add, one FMA per product in k order.
//
// The kernel for A and B that TMA can describe (16-byte aligned bases and
// row pitches).  What it keeps from the pages and what changes for GB300:
//   * Block tile 128 x 128, K slices of 32, register tiling of 8 x 16
//     outputs per thread ("SGEMM CUDA代码学习", "第 2 步"; "CUDA GEMM：从基础
//     写法到工程优化", "5. 2D Block Tiling") and warp tiles of 64 x 64 ("10.
//     Warp Tiling"): four warps, 2 x 2.
//   * Staging: one thread issues two 2-D TMA copies per K slice -- A's
//     128 x 32 box and B's 32 x 128 box -- into a 3-stage ring; an mbarrier
//     per stage counts the bytes.  No thread spends instructions on loads or
//     address arithmetic, and no __syncthreads sits in the main loop.  This
//     is the multi-stage asynchronous copy of "第 5 步" / "12. Async Copy
//     Double Buffering" in its Blackwell form.
//   * Bank conflicts: A stays row-major in shared memory (no transposing
//     copy) under TMA's 128-byte swizzle -- 16-byte chunk c of row r lives
//     at chunk c ^ (r mod 8), the hardware form of the XOR swizzle of "HGEMM
//     SMEM Swizzle 代码学习".  A thread reads four consecutive k of one row
//     with one 16-byte load; the eight rows a warp reads together are eight
//     consecutive rows, so they land in eight distinct bank groups.  B rows
//     are read as 16-byte pieces of 64 contiguous bytes per warp.
//   * No producer warp: the warp whose arrival completes a stage's count
//     (a shared-memory counter) issues that stage's refill.  Four warps per
//     CTA and two CTAs per SM keep two warps on each SM sub-partition, each
//     with up to 255 registers.
//   * The FMAs are Blackwell's packed two-lane form (fma.rn.f32x2), issued
//     column-pair-major: one pair of B values meets eight rows of A in eight
//     consecutive instructions.  Every output still gets one FP32 FMA per k,
//     in k order, so results are bit-identical to the cp.async kernel.
//   * Tails: TMA reads zeros outside M, N and K; the epilogue masks rows and
//     columns outside C.  Epilogue alpha * acc + beta * C_old, C not read
//     when beta == 0, 16-byte stores where C allows.
//   * Every mbarrier wait is bounded; a wait that runs out records
//     DGEMM_ERR_TIMEOUT in this file's device status word, the CTA stops,
//     and one thread waits (again bounded) for the copies it issued before
//     the CTA leaves.
#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dgemm.h"
#include "internal.h"
#include "ptx.cuh"

#define DGEMM_UNIT 2
#include "checked.cuh"

namespace dgemm {

__device__ int g_simt_status;

namespace {

constexpr int BM = 128;
constexpr int BK = 32;                              // K per stage: one 128-byte row of A
constexpr int A_TILE_BYTES = BM * BK * 4;           // 16 KB
constexpr int kGroupM = 16;                         // rasterisation group height, in tiles
constexpr uint64_t kWaitLimitNs = 4000000000ull;    // 4 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;   // 1 s

// Thread and warp tiling.  LM x LN lanes (LM * LN = 32): a thread holds the
// 8 rows ty + LM * i (i < 8) and TNG groups of 4 columns tx * 4 + 4 * LN * h
// (h < TNG) of its warp's tile; WGM x WGN warps.
template <int LM, int TNG, int WGM, int WGN, int STAGES>
struct TmaShape {
    static constexpr int LN = 32 / LM;
    static constexpr int WTM = 8 * LM, WTN = 4 * LN * TNG;
    static constexpr int BN = WGN * WTN, WARPS = WGM * WGN, THREADS = 32 * WARPS;
    static constexpr int B_TILE_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static_assert(WGM * WTM == BM, "128 rows per tile");
    static_assert(BN <= 256, "B comes as one TMA box per stage");
    static_assert(STAGE_BYTES % 1024 == 0, "stages start on the swizzle pattern's 1024-byte period");
};

// The configuration in use: 128 x 128 tiles, 8 x 16 outputs per thread.
using Cfg = TmaShape<8, 4, 2, 2, 3>;
constexpr int kMinBlocks = 2;

struct TmaCtl {
    uint64_t full[8];  // stage landed (TMA transaction bytes)
    uint64_t never;    // test hook: a barrier nothing arrives at
    int cnt[8];        // warps done with the stage
    int abort;         // a wait ran out: every warp stops
    int issued;        // K slices whose copies have been issued
};
static_assert(Cfg::RING_BYTES + 1024 + static_cast<int>(sizeof(TmaCtl)) <= 113 * 1024,
              "two CTAs fit in one SM's shared memory");
constexpr int kSmemBytes = Cfg::RING_BYTES + 1024 + static_cast<int>(sizeof(TmaCtl));

struct TmaParams {
    int64_t M, N, K;
    float alpha, beta;
    float *C;
    int64_t ldc;
    int vec_c;         // C's base and pitch allow 16-byte stores
    int inject_stall;  // test hook: wait on `never` first, so the waits run out
    uint64_t wait_limit_ns;
    int64_t m_checked;  // rows of C the checked build lets the stores reach (M unless a test shrinks it)
};

__device__ __forceinline__ bool aborted(const int *abort)
{
    return *reinterpret_cast<const volatile int *>(abort) != 0;
}

// The slow part of wait_phase: poll until the phase completes, the limit
// runs out (which raises the abort flag and records DGEMM_ERR_TIMEOUT) or
// another warp raised the flag.  Inlined: a call inside the main loop would
// constrain the register allocation of the ~210 registers live there.
__device__ __forceinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, int *abort, uint64_t limit_ns)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (aborted(abort)) return false;
        if (ptx::globaltimer_ns() - t0 > limit_ns) {
            atomicCAS(&g_simt_status, 0, DGEMM_ERR_TIMEOUT);
            *reinterpret_cast<volatile int *>(abort) = 1;
            return false;
        }
    }
}

// Bounded wait for the phase of the given parity; false on time-out or
// abort (see wait_phase_slow).  The first probe is inline: a stage that has
// already landed costs one try_wait.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, int *abort, uint64_t limit_ns)
{
    return ptx::mbar_try_wait(bar, parity) || wait_phase_slow(bar, parity, abort, limit_ns);
}

// Issue K slice kt into `stage`: arm the stage's barrier with the bytes of
// both boxes, then A's 128 x 32 box at (kt * 32, m0) and B's 32 x BN box at
// (n0, kt * 32).  Boxes that reach past M, N or K are filled with zeros.
__device__ __forceinline__ void issue_slice(uint32_t ring, TmaCtl *ctl, int stage, int64_t kt, int64_t m0,
                                            int64_t n0, const CUtensorMap *ta, const CUtensorMap *tb)
{
    const uint32_t full = ptx::smem_addr(&ctl->full[stage]);
    ptx::mbar_arrive_expect_tx(full, Cfg::STAGE_BYTES);
    const uint32_t sa = ring + static_cast<uint32_t>(stage) * Cfg::STAGE_BYTES;
    const int32_t k0 = static_cast<int32_t>(kt * BK);
    ptx::tma_load_2d(sa, ta, full, k0, static_cast<int32_t>(m0));
    ptx::tma_load_2d(sa + A_TILE_BYTES, tb, full, static_cast<int32_t>(n0), k0);
}

__device__ __forceinline__ void store4(float *__restrict__ p, int64_t gn, int64_t N, const float (&o)[4], float beta,
                                       bool vec)
{
    // (columns at or past N are masked below: the last tile column may reach past C)
    if (vec && gn + 3 < N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(p) & 15u) == 0)) {
        float4 v = make_float4(o[0], o[1], o[2], o[3]);
        if (beta != 0.f) {
            const float4 c = *reinterpret_cast<const float4 *>(p);
            v.x = fmaf(beta, c.x, v.x);
            v.y = fmaf(beta, c.y, v.y);
            v.z = fmaf(beta, c.z, v.z);
            v.w = fmaf(beta, c.w, v.w);
        }
        *reinterpret_cast<float4 *>(p) = v;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (gn + j < N) p[j] = beta != 0.f ? fmaf(beta, p[j], o[j]) : o[j];
    }
}

template <int LM, int TNG, int WGM, int WGN, int STAGES>
__global__ void __launch_bounds__(TmaShape<LM, TNG, WGM, WGN, STAGES>::THREADS, kMinBlocks)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const TmaParams p)
{
    using S = TmaShape<LM, TNG, WGM, WGN, STAGES>;
    constexpr int LN = S::LN, BN = S::BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
    TmaCtl *ctl = reinterpret_cast<TmaCtl *>(smem_raw + (ring - raw) + S::RING_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Grouped rasterisation: runs of kGroupM consecutive CTAs walk down M
    // inside one column of tiles, so CTAs resident together share B columns
    // and a short band of A rows in L2.
    int64_t m0, n0;
    {
        const int64_t b = blockIdx.x;
        const int64_t tiles_m = (p.M + BM - 1) / BM;
        const int64_t per_group = static_cast<int64_t>(kGroupM) * ((p.N + BN - 1) / BN);
        const int64_t g = b / per_group, r = b % per_group;
        const int64_t gm = tiles_m - g * kGroupM < kGroupM ? tiles_m - g * kGroupM : kGroupM;
        m0 = (g * kGroupM + r % gm) * BM;
        n0 = (r / gm) * BN;
    }
    const int64_t num_kt = (p.K + BK - 1) / BK;
    const uint64_t limit = p.wait_limit_ns;
    // the raster is a bijection onto the tiles: no CTA's tile starts outside C
    const bool tile_ok = DGEMM_CHECK(m0 >= 0 && m0 < p.M && n0 >= 0 && n0 < p.N);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctl->full[s]), 1);
            ctl->cnt[s] = 0;
        }
        ptx::mbar_init(ptx::smem_addr(&ctl->never), 1);
        ctl->abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
        const int first = num_kt < STAGES ? static_cast<int>(num_kt) : STAGES;
        for (int s = 0; s < first; ++s) issue_slice(ring, ctl, s, s, m0, n0, &tmap_a, &tmap_b);
        ctl->issued = first;
    }
    __syncthreads();

    const int wm = warp / WGN, wn = warp % WGN;
    const int ty = lane / LN, tx = lane % LN;
    float2 acc[8][2 * TNG];  // acc[i][j]: row i, columns 2j and 2j + 1 of the thread's 4 * TNG
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 2 * TNG; ++j) acc[i][j] = make_float2(0.f, 0.f);
    const uint32_t a_off = static_cast<uint32_t>((wm * S::WTM + ty) * 128);
    const uint32_t b_off = static_cast<uint32_t>(A_TILE_BYTES + (wn * S::WTN + tx * 4) * 4);
    // every fragment read stays inside its stage: A rows < 128, 16-byte
    // chunks < 8; B columns + the last group's 4 < BN
    const bool frag_ok = DGEMM_CHECK(a_off + 7 * LM * 128 + 7 * 16 + 16 <= static_cast<uint32_t>(A_TILE_BYTES) &&
                                     b_off + (BK - 1) * BN * 4 + (TNG - 1) * LN * 16 + 16 <=
                                         static_cast<uint32_t>(S::STAGE_BYTES));

    // (warp-uniform: the loop below holds warp-collective votes)
    bool ok = __all_sync(0xffffffffu, tile_ok && frag_ok);
    if (!ok) *reinterpret_cast<volatile int *>(&ctl->abort) = 1;  // a failed check: stop, and drain the copies
    if (ok && p.inject_stall)
        ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&ctl->never), 0, &ctl->abort, limit));
    uint32_t phase = 0;
    int stage = 0;
    for (int64_t kt = 0; ok && kt < num_kt; ++kt) {
        ok = __all_sync(0xffffffffu, wait_phase(ptx::smem_addr(&ctl->full[stage]), phase, &ctl->abort, limit));
        if (!ok) break;
        const uint32_t sa = ring + static_cast<uint32_t>(stage) * S::STAGE_BYTES + a_off;
        const uint32_t sb = ring + static_cast<uint32_t>(stage) * S::STAGE_BYTES + b_off;
#pragma unroll
        for (int kc = 0; kc < BK / 4; ++kc) {
            // rows ty + LM * i, k = 4 kc .. 4 kc + 3: 16-byte chunk kc of the
            // row sits at chunk kc ^ (row mod 8)
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                a[i] = ptx::ld_shared_v4f(sa + i * LM * 128 +
                                          static_cast<uint32_t>((kc ^ ((ty + LM * i) & 7)) << 4));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int k = kc * 4 + kk;
                float2 bp[2 * TNG];
#pragma unroll
                for (int h = 0; h < TNG; ++h) {
                    const float4 b = ptx::ld_shared_v4f(sb + k * BN * 4 + h * LN * 16);
                    bp[2 * h] = make_float2(b.x, b.y);
                    bp[2 * h + 1] = make_float2(b.z, b.w);
                }
#pragma unroll
                for (int j = 0; j < 2 * TNG; ++j)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                        acc[i][j] = __ffma2_rn(make_float2(av, av), bp[j], acc[i][j]);
                    }
            }
        }
        // this warp is done with the stage; the warp that completes the
        // count refills it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&ctl->cnt[stage], 1) == S::WARPS - 1) {
                ctl->cnt[stage] = 0;
                __threadfence_block();
                if (kt + STAGES < num_kt && !aborted(&ctl->abort)) {
                    issue_slice(ring, ctl, stage, kt + STAGES, m0, n0, &tmap_a, &tmap_b);
                    ctl->issued = static_cast<int>(kt + STAGES + 1);
                }
            }
        }
        if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
        }
    }

    if (ok) {
        const bool vec = p.vec_c != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t gm = m0 + wm * S::WTM + ty + LM * i;
            if (gm >= p.M) continue;
            if (!DGEMM_CHECK(gm < p.m_checked)) continue;
#pragma unroll
            for (int h = 0; h < TNG; ++h) {
                const int64_t gn = n0 + wn * S::WTN + h * LN * 4 + tx * 4;
                const float o[4] = {p.alpha * acc[i][2 * h].x, p.alpha * acc[i][2 * h].y,
                                    p.alpha * acc[i][2 * h + 1].x, p.alpha * acc[i][2 * h + 1].y};
                store4(p.C + gm * p.ldc + gn, gn, p.N, o, p.beta, vec);
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && aborted(&ctl->abort)) {
        // Do not leave while TMA may still write this CTA's shared memory:
        // wait (bounded) for the last copies issued to each stage.
        const int issued = *reinterpret_cast<volatile int *>(&ctl->issued);
        for (int kt = issued - STAGES < 0 ? 0 : issued - STAGES; kt < issued; ++kt) {
            const uint32_t bar = ptx::smem_addr(&ctl->full[kt % STAGES]);
            const uint32_t parity = static_cast<uint32_t>(kt / STAGES) & 1u;
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar, parity))
                if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) break;
        }
    }
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, TmaParams);
constexpr KernelFn kKernel = sgemm_tma_kernel<8, 4, 2, 2, 3>;

// Sets the kernel's shared-memory limit once per device; false if refused.
bool kernel_ready()
{
    constexpr int kMaxDevices = 64;
    static bool ok[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::call_once(once[dev], [dev] {
        ok[dev] = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) ==
                  cudaSuccess;
        if (!ok[dev]) cudaGetLastError();
    });
    return ok[dev];
}

}  // namespace

const char *launch_sgemm_tma(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float beta, float *C, int64_t ldc, cudaStream_t stream)
{
    // TMA coordinates are 32-bit; the caller has checked alignment
    constexpr int64_t kCoordMax = (int64_t(1) << 31) - 256;
    if (M > kCoordMax || N > kCoordMax || K > kCoordMax) return nullptr;
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + Cfg::BN - 1) / Cfg::BN);
    if (tiles > INT32_MAX) return nullptr;  // (a C of 2^45 elements: no GPU holds one)
    CUtensorMap ma, mb;
    if (!encode_tiled_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, static_cast<uint64_t>(K),
                         static_cast<uint64_t>(M), static_cast<uint64_t>(lda) * 4, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, B, static_cast<uint64_t>(N),
                         static_cast<uint64_t>(K), static_cast<uint64_t>(ldb) * 4, Cfg::BN, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
        return nullptr;
    if (!kernel_ready()) return nullptr;
    TmaParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.vec_c = aligned16(C) && (ldc % 4 == 0) ? 1 : 0;
    const uint64_t stall = take_injected_stall();
    p.inject_stall = stall ? 1 : 0;
    p.wait_limit_ns = stall ? stall : kWaitLimitNs;
    const int64_t shrink = take_shrink_bounds();
    p.m_checked = shrink < M ? M - shrink : 0;
    kKernel<<<static_cast<unsigned>(tiles), Cfg::THREADS, kSmemBytes, stream>>>(ma, mb, p);
    return "sgemm_simt_tma_128x128x32_ffma2";
}

int simt_read_status(int clear)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_simt_status, sizeof(int)) != cudaSuccess) return DGEMM_ERR_LAUNCH;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_simt_status, &zero, sizeof(int)) != cudaSuccess) return DGEMM_ERR_LAUNCH;
    }
    return v;
}

}  // namespace dgemm

DGEMM_DEFINE_CHECK_READER(check_status_tma)
