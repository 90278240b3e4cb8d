// umma_gemm.cu -- tensor-core GEMM for sm_103a on tcgen05 (5th-generation
// tensor cores, accumulators in tensor memory), for two input types:
//
//   FP16 TN : C(f16) = alpha * A * B^T + beta * C, A M x K and B N x K
//             row-major (both K-major), FP32 accumulation;
//   TF32    : C(f32) = alpha * A * B + beta * C, A M x K (K-major) and
//             B K x N row-major (N-major), operands read as TF32.
//
// Structure -- a persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: one thread streams 128 x BK tiles of A and
//               BK x 256 tiles of B into a 4-stage shared-memory ring
//               (128-byte swizzled rows), signalling "full" mbarriers with
//               transaction byte counts;
//   warp 1      MMA issuer: one thread waits for a full stage, issues
//               BK/UMMA_K tcgen05.mma instructions of 128 x 256 x UMMA_K into
//               a TMEM accumulator, and commits the stage back to its
//               "empty" mbarrier when those MMAs have read it;
//   warps 2..5  epilogue: drain the accumulator TMEM -> registers
//               (tcgen05.ld), form alpha * acc + beta * C_old in FP32 and
//               store with 16-byte vectors, masked at the M / N edges.
// Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile run
// while the MMAs of the next tile proceed.
//
// This is the GB300 form of the pages' designs:
//   * the producer / consumer split with a stage ring and acquire / release
//     primitives -- "Warp Specialization HGEMM", sections "1. 角色划分" to
//     "4. consumer 的双重流水" (cuda::pipeline there, mbarriers here);
//   * the XOR smem swizzle of "HGEMM SMEM Swizzle 代码学习" ("swizzle 核心"),
//     here the hardware 128-byte swizzle written by TMA and read by the MMA
//     through the matching descriptor mode;
//   * the multi-stage async-copy ring of "SGEMM CUDA代码学习", "第 5 步"
//     (cp.async + wait_group there, TMA + mbarrier transaction counts here);
//   * block-order swizzling for L2 reuse ("第 5 步", block swizzle), here the
//     persistent scheduler's grouped tile order.
// Tails: TMA fills out-of-range rows / columns / K with zeros, which add
// exact zeros to the sums, and the epilogue masks stores outside M x N.
//
// Every mbarrier wait is bounded (a few seconds of %globaltimer): a wait that
// runs out records DGEMM_ERR_TIMEOUT in the device status word, raises an
// abort flag that the other roles also poll, waits (again bounded) for its
// own copies and MMAs in flight, and the CTA releases its TMEM and exits.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <mutex>
#include <string>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dgemm.h"
#include "internal.h"
#include "ptx.cuh"

#define DGEMM_UNIT 3
#include "checked.cuh"

namespace dgemm {

__device__ int g_umma_status;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int STAGES = 4;
// The TMA-fed single-CTA kernel sizes its ring at run time: stages of
// A_TILE_BYTES + bn * ROW_BYTES, as many as fit (at most MAX_STAGES) --
// narrow tiles keep more bytes in flight.  The non-TMA producers use STAGES
// stages of STAGE_BYTES.
constexpr int ROW_BYTES = 128;                     // one swizzled row
constexpr int A_TILE_BYTES = BM * ROW_BYTES;       // 16 KB
constexpr int B_TILE_BYTES = BN * ROW_BYTES;       // 32 KB
constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int MAX_STAGES = 8;
constexpr int TMEM_COLS = 2 * BN;                  // two f32 accumulators
constexpr int kGroupN = 8;                         // tile-order group width
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s, default wait bound
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // 1 s

// Operand kinds.  TN: B stored N x K (K-major); NN: B stored K x N
// (N-major).  TF32 reads FP32 storage; all kinds accumulate in FP32.
enum { kF16 = 0, kTF32 = 1, kBF16 = 2, kF16NN = 3, kBF16NN = 4 };

template <int kKind>
struct Traits {
    static constexpr bool kTf32 = kKind == kTF32;
    static constexpr int kElem = kTf32 ? 4 : 2;         // bytes per A / B / C element
    static constexpr int BK = ROW_BYTES / kElem;         // K per stage: one 128-byte row
    static constexpr int UMMA_K = 32 / kElem;            // K per MMA: 32 bytes
    static constexpr bool kBF = kKind == kBF16 || kKind == kBF16NN;
    // B stored K x N (N-major) rather than N x K
    static constexpr bool kBNMajor = kKind == kTF32 || kKind == kF16NN || kKind == kBF16NN;
    // operand format code of the instruction descriptor: f16 0, bf16 1, tf32 2
    static constexpr uint32_t kFmt = kTf32 ? 2u : (kBF ? 1u : 0u);
    // N-major B in shared memory: boxes of 128 bytes of columns x BK rows.
    // 16-bit: 128-byte swizzle of 16-byte chunks, 8-row K groups 1 KB apart;
    // 32-bit: the 32-byte-chunk swizzle, read as 4-row halves 512 B apart.
    static constexpr int kNBox = ROW_BYTES / kElem;       // columns per box: 64 or 32
    static constexpr uint32_t kNBoxBytes = BK * ROW_BYTES;  // 8 KB or 4 KB
    static constexpr uint32_t kNLayout = kTf32 ? ptx::kSw128A32 : ptx::kSw128;
    static constexpr uint32_t kNSbo = kTf32 ? 512u : 1024u;
    static constexpr uint32_t kNStep = UMMA_K * ROW_BYTES;  // bytes of one MMA's K rows
    // D = f32 (bits 4-5 = 1), A / B formats, B major (bit 16), N >> 3, M >> 4
    static constexpr uint32_t kIdesc = (1u << 4) | (kFmt << 7) | (kFmt << 10) |
                                       ((kBNMajor ? 1u : 0u) << 16) |
                                       (static_cast<uint32_t>(BN >> 3) << 17) |
                                       (static_cast<uint32_t>(BM >> 4) << 24);
    // B staged K-major (the register-path producers transpose it)
    static constexpr uint32_t kIdescKMajorB = kIdesc & ~(1u << 16);
};

// 2-byte output conversions (f16 or bf16), round to nearest even.
template <bool kBF>
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    if constexpr (kBF) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

template <bool kBF>
__device__ __forceinline__ float2 unpack2(uint32_t u)
{
    if constexpr (kBF)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
    else
        return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}

template <bool kBF>
__device__ __forceinline__ float load1(const uint16_t *p)
{
    const uint16_t u = *p;
    if constexpr (kBF)
        return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(&u));
    else
        return __half2float(*reinterpret_cast<const __half *>(&u));
}

template <bool kBF>
__device__ __forceinline__ uint16_t round1(float v)
{
    if constexpr (kBF) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<const uint16_t *>(&h);
    } else {
        const __half h = __float2half_rn(v);
        return *reinterpret_cast<const uint16_t *>(&h);
    }
}

// Per-CTA wait control: the abort flag every role polls and the wait limit.
struct WaitCtl {
    int abort;
    int pad;
    uint64_t limit_ns;
};

struct Ctrl {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint64_t never;  // test hook: a barrier nothing arrives at
    WaitCtl wait;
    uint32_t tmem_base;
};



struct Params {
    int64_t M, N, K;
    float alpha, beta;
    void *C;
    int64_t ldc;
    int64_t tiles_m, tiles_n, num_kb;
    int vec_c;
    // operands for the register-path producer (unused with TMA)
    const void *A;
    const void *B;
    int64_t lda, ldb;
    // bound of every mbarrier wait, and the test-only fault injection: when
    // set, the MMA issuer first waits on a barrier nothing arrives at, so the
    // waits run out
    uint64_t wait_limit_ns;
    int inject_stall;
    // split-K: the S CTAs of a cluster share one output tile, each summing a
    // contiguous range of K blocks (1 = no split)
    int splitk;
    // epilogue stores C through shared-memory boxes and TMA (else direct
    // 16-byte / scalar stores)
    int tma_store;
    // output tile width of the single-CTA TMA kernel: a multiple of 32 (of 64
    // for 16-bit N-major B) from 32 to 256; the CTA-pair and register-path
    // kernels use 256.  The MMA is 128 x bn x UMMA_K.
    int bn;
    // single-CTA kernel: stages in its ring and bytes per stage (1024-byte
    // multiples).  The TMA producer fills a stage with kpb K blocks (1 or 2),
    // each A_TILE_BYTES of A then bn * ROW_BYTES of B; the non-TMA producers
    // use one K block of STAGE_BYTES
    int stages, stage_bytes, kpb;
    // CTA-pair kernel with N-major B: the stage's B half comes as one 3-D box
    // (column group of 128 bytes x BK rows x 128 / kNBox groups) instead of
    // 128 / kNBox 2-D boxes.  The 3-D map covers columns [0, b3d_cols) -- the
    // whole column groups; a half that reaches past them (the last tile
    // column, when N is not a whole number of groups) takes the 2-D boxes of
    // the second map
    int b3d;
    int64_t b3d_cols;
    // CTA-pair kernel, stream-K: tiles [0, sk_tiles) of the tile order are
    // cut along K into one contiguous range of K blocks per pair (0 = every
    // tile whole).  A pair that ends inside a tile leaves its raw partial
    // accumulator in its slot of sk_work and stamps sk_flags with sk_gen; the
    // pair that continues the tile loads it into TMEM and keeps accumulating.
    int64_t sk_tiles;
    float *sk_work;
    uint64_t *sk_flags;
    uint64_t sk_gen;
};

// The instruction descriptor with its N field (bits 17-22, N >> 3) set to n.
__device__ __forceinline__ uint32_t idesc_with_n(uint32_t idesc, int n)
{
    return (idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(n >> 3) << 17);
}

__device__ __forceinline__ void tile_coords(int64_t t, const Params &p, int64_t &m0, int64_t &n0,
                                            int64_t bm = BM)
{
    // Groups of kGroupN tile columns; inside a group consecutive tiles share
    // one A row band and walk N, so the tiles in flight at once read a few
    // B column bands and a few A row bands.
    const int64_t per_group = static_cast<int64_t>(kGroupN) * p.tiles_m;
    const int64_t g = t / per_group, r = t % per_group;
    const int64_t left = p.tiles_n - g * kGroupN;
    const int64_t gn = left < kGroupN ? left : kGroupN;
    n0 = (g * kGroupN + r % gn) * p.bn;
    m0 = (r / gn) * bm;
}

// The work of one CTA: tiles t0, t0 + dt, ... and, with split-K, the K
// blocks [kb0, kb1) of each (the S CTAs of a cluster share a tile; rank r
// takes the r-th of S near-equal contiguous ranges).
struct Sched {
    int64_t t0, dt, kb0, kb1;
};

__device__ __forceinline__ Sched schedule(const Params &p)
{
    Sched s;
    const int S = p.splitk;
    if (S > 1) {
        const int64_t r = ptx::cluster_ctarank();
        s.t0 = blockIdx.x / S;
        s.dt = gridDim.x / S;
        s.kb0 = r * p.num_kb / S;
        s.kb1 = (r + 1) * p.num_kb / S;
    } else {
        s.t0 = blockIdx.x;
        s.dt = gridDim.x;
        s.kb0 = 0;
        s.kb1 = p.num_kb;
    }
    return s;
}

__device__ __forceinline__ bool aborted(const WaitCtl *wc)
{
    return *reinterpret_cast<const volatile int *>(&wc->abort) != 0;
}

__device__ __forceinline__ void raise_abort(WaitCtl *wc)
{
    if (atomicExch(&g_umma_status, DGEMM_ERR_TIMEOUT) == 0) __threadfence();
    *reinterpret_cast<volatile int *>(&wc->abort) = 1;
}

// Bounded wait for the phase of the given parity; false on time-out or when
// another role raised the abort flag.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, WaitCtl *wc)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns(), limit = wc->limit_ns;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (aborted(wc)) return false;
        if (ptx::globaltimer_ns() - t0 > limit) {
            raise_abort(wc);
            return false;
        }
    }
}

// Same, with cluster-scope acquire (barriers that the other CTA of a pair
// arrives on, directly or through a multicast commit).
__device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity, WaitCtl *wc)
{
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns(), limit = wc->limit_ns;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if (aborted(wc)) return false;
        if (ptx::globaltimer_ns() - t0 > limit) {
            raise_abort(wc);
            return false;
        }
    }
}

// Bounded wait used on the way out, after an abort: ignores the abort flag.
__device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer_ns() - t0 > kDrainLimitNs) return false;
    return true;
}

template <int kKind, int kKpb>
__device__ __forceinline__ void run_producer(const CUtensorMap *tmap_a, const CUtensorMap *tmap_b,
                                             const Params &p, uint32_t smem_base, Ctrl *ctrl,
                                             WaitCtl *wc)
{
    using T = Traits<kKind>;
    const int64_t num_tiles = p.tiles_m * p.tiles_n;
    const Sched sc = schedule(p);
    uint32_t stage = 0, phase = 0;
    uint32_t issued = 0, issued_phase = 0;  // per-stage: a load was issued / its phase
    bool ok = true;
    for (int64_t t = sc.t0; ok && t < num_tiles; t += sc.dt) {
        int64_t m0, n0;
        tile_coords(t, p, m0, n0);
        for (int64_t kb = sc.kb0; kb < sc.kb1; kb += kKpb) {
            if (!wait_bounded(ptx::smem_addr(&ctrl->empty[stage]), phase ^ 1u, wc)) {
                ok = false;
                break;
            }
            // K blocks kb and (two per stage, if inside the range) kb + 1,
            // one after the other in the stage
            const bool second = kKpb == 2 && kb + 1 < sc.kb1;
            const uint32_t half = A_TILE_BYTES + static_cast<uint32_t>(p.bn) * ROW_BYTES;
            const uint32_t full = ptx::smem_addr(&ctrl->full[stage]);
            ptx::mbar_arrive_expect_tx(full, second ? 2 * half : half);
#pragma unroll
            for (int h = 0; h < kKpb; ++h) {
                if (h == 1 && !second) break;
                const uint32_t sa = smem_base + stage * static_cast<uint32_t>(p.stage_bytes) + h * half;
                const uint32_t sb = sa + A_TILE_BYTES;
                const int32_t kc = static_cast<int32_t>((kb + h) * T::BK);
                ptx::tma_load_2d(sa, tmap_a, full, kc, static_cast<int32_t>(m0));
                if constexpr (!T::kBNMajor) {
                    ptx::tma_load_2d(sb, tmap_b, full, kc, static_cast<int32_t>(n0));
                } else if (p.b3d) {
                    // B is N-major, all bn / kNBox column groups in one 3-D box
                    ptx::tma_load_3d(sb, tmap_b, full, 0, kc, static_cast<int32_t>(n0 / T::kNBox));
                } else {
                    // B is N-major: boxes of 128 bytes of columns x BK rows, one
                    // swizzle column each (see Traits)
#pragma unroll 1
                    for (int c = 0; c < p.bn / T::kNBox; ++c)
                        ptx::tma_load_2d(sb + c * T::kNBoxBytes, tmap_b, full,
                                         static_cast<int32_t>(n0 + c * T::kNBox), kc);
                }
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == static_cast<uint32_t>(p.stages)) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        // Do not leave while TMA may still be writing into this CTA's smem.
        for (int s = 0; s < p.stages; ++s)
            if ((issued >> s) & 1u)
                drain_wait(ptx::smem_addr(&ctrl->full[s]), (issued_phase >> s) & 1u);
    }
}

// Byte offset of (row r, byte b of the row) in a K-major tile of 128-byte
// rows under the 128-byte swizzle: 16-byte chunk j of row r is stored at
// chunk position j ^ (r mod 8).  This is the placement TMA's 128-byte swizzle
// writes, so both producers feed the same MMA descriptors.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t b)
{
    return r * 128u + ((((b >> 4) ^ (r & 7u)) << 4) | (b & 15u));
}

template <typename E>
__device__ __forceinline__ void st_shared(uint32_t addr, E v)
{
    if constexpr (sizeof(E) == 2)
        asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
    else
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Register-path producer for operands TMA cannot describe (base pointers or
// row pitches that are not 16-byte aligned): 128 threads load elements with
// plain predicated loads (zeros outside M, N, K), write them into the same
// swizzled K-major tiles -- transposing an N-major B on the way -- then make
// the writes visible to the tensor core (proxy fence) and arrive on the
// stage's "full" barrier (128 arrivals).
template <int kKind>
__device__ __forceinline__ void run_reg_producer(const Params &p, uint32_t smem_base, Ctrl *ctrl,
                                                 int ptid, WaitCtl *wc)
{
    using T = Traits<kKind>;
    using E = typename std::conditional<T::kElem == 2, uint16_t, uint32_t>::type;
    constexpr int BK = T::BK;
    constexpr int kBatch = 8;
    const E *__restrict__ A = static_cast<const E *>(p.A);
    const E *__restrict__ B = static_cast<const E *>(p.B);
    const int64_t num_tiles = p.tiles_m * p.tiles_n;
    const Sched sc = schedule(p);
    uint32_t stage = 0, phase = 0;
    for (int64_t t = sc.t0; t < num_tiles; t += sc.dt) {
        int64_t m0, n0;
        tile_coords(t, p, m0, n0);
        for (int64_t kb = sc.kb0; kb < sc.kb1; ++kb) {
            if (!wait_bounded(ptx::smem_addr(&ctrl->empty[stage]), phase ^ 1u, wc)) return;
            const int64_t k0 = kb * BK;
            const uint32_t sa = smem_base + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_TILE_BYTES;
            // A tile: BM rows x BK; consecutive threads take consecutive k.
            for (int i0 = 0; i0 < BM * BK / 128; i0 += kBatch) {
                E v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int idx = ptid + (i0 + u) * 128;
                    const int64_t gm = m0 + idx / BK, gk = k0 + idx % BK;
                    v[u] = (gm < p.M && gk < p.K) ? A[gm * p.lda + gk] : E(0);
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int idx = ptid + (i0 + u) * 128;
                    const uint32_t off = sw128_offset(idx / BK, (idx % BK) * sizeof(E));
                    if (DGEMM_CHECK(off + sizeof(E) <= static_cast<uint32_t>(A_TILE_BYTES))) st_shared(sa + off, v[u]);
                }
            }
            // B tile, staged K-major: row n holds BK consecutive k.
            for (int i0 = 0; i0 < BN * BK / 128; i0 += kBatch) {
                E v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int idx = ptid + (i0 + u) * 128;
                    if constexpr (!T::kBNMajor) {  // B stored N x K: walk k
                        const int64_t gn = n0 + idx / BK, gk = k0 + idx % BK;
                        v[u] = (gn < p.N && gk < p.K) ? B[gn * p.ldb + gk] : E(0);
                    } else {  // B stored K x N: walk n (coalesced), transpose into smem
                        const int64_t gn = n0 + idx % BN, gk = k0 + idx / BN;
                        v[u] = (gn < p.N && gk < p.K) ? B[gk * p.ldb + gn] : E(0);
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int idx = ptid + (i0 + u) * 128;
                    const int n = !T::kBNMajor ? idx / BK : idx % BN;
                    const int k = !T::kBNMajor ? idx % BK : idx / BN;
                    const uint32_t off = sw128_offset(n, k * sizeof(E));
                    if (DGEMM_CHECK(off + sizeof(E) <= static_cast<uint32_t>(B_TILE_BYTES))) st_shared(sb + off, v[u]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_addr(&ctrl->full[stage]));
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// cp.async producer for 4-byte operands (TF32) that TMA cannot describe:
// the same swizzled K-major tiles as run_reg_producer, but every element is a
// 4-byte asynchronous copy (zero-filled outside M, N, K), so each thread keeps
// kInFlight stages of copies outstanding instead of waiting for its loads.
// A stage's "full" barrier gets this thread's arrival once its copies of
// that stage have landed (cp.async.wait_group) and been fenced to the async
// proxy.  kInFlight < STAGES, so the MMA can always drain the oldest stage.
__device__ __forceinline__ void cp_async4_zfill(uint32_t dst, const void *src, bool ok)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0)
                 : "memory");
}

template <int kPending>
__device__ __forceinline__ void cp_async_wait_pending()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

__device__ __forceinline__ void run_cpasync_producer(const Params &p, uint32_t smem_base, Ctrl *ctrl,
                                                     int ptid, WaitCtl *wc)
{
    using T = Traits<kTF32>;
    constexpr int BK = T::BK;
    constexpr int kInFlight = 3;
    static_assert(kInFlight < STAGES, "the oldest stage must be released before a slot is reused");
    const float *__restrict__ A = static_cast<const float *>(p.A);
    const float *__restrict__ B = static_cast<const float *>(p.B);
    const int64_t num_tiles = p.tiles_m * p.tiles_n;
    const Sched sc = schedule(p);
    uint32_t stage = 0, phase = 0;
    uint32_t pending[kInFlight];
    int npending = 0;
    bool ok = true;
    for (int64_t t = sc.t0; ok && t < num_tiles; t += sc.dt) {
        int64_t m0, n0;
        tile_coords(t, p, m0, n0);
        for (int64_t kb = sc.kb0; kb < sc.kb1; ++kb) {
            if (!wait_bounded(ptx::smem_addr(&ctrl->empty[stage]), phase ^ 1u, wc)) {
                ok = false;
                break;
            }
            const int64_t k0 = kb * BK;
            const uint32_t sa = smem_base + stage * STAGE_BYTES;
            const uint32_t sb = sa + A_TILE_BYTES;
            // A tile: BM rows x BK; consecutive threads take consecutive k
#pragma unroll 8
            for (int i = 0; i < BM * BK / 128; ++i) {
                const int idx = ptid + i * 128;
                const int r = idx / BK, c = idx % BK;
                const int64_t gm = m0 + r, gk = k0 + c;
                const bool in = gm < p.M && gk < p.K;
                if (DGEMM_CHECK(sw128_offset(r, c * 4) + 4 <= static_cast<uint32_t>(A_TILE_BYTES)))
                    cp_async4_zfill(sa + sw128_offset(r, c * 4), in ? A + gm * p.lda + gk : A, in);
            }
            // B tile (stored K x N): consecutive threads take consecutive n;
            // staged K-major (row n holds BK consecutive k)
#pragma unroll 8
            for (int i = 0; i < BN * BK / 128; ++i) {
                const int idx = ptid + i * 128;
                const int n = idx % BN, k = idx / BN;
                const int64_t gn = n0 + n, gk = k0 + k;
                const bool in = gn < p.N && gk < p.K;
                if (DGEMM_CHECK(sw128_offset(n, k * 4) + 4 <= static_cast<uint32_t>(B_TILE_BYTES)))
                    cp_async4_zfill(sb + sw128_offset(n, k * 4), in ? B + gk * p.ldb + gn : B, in);
            }
            ptx::cp_async_commit_group();
            pending[npending++] = stage;
            if (npending == kInFlight) {
                cp_async_wait_pending<kInFlight - 1>();  // the oldest stage's copies landed
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(ptx::smem_addr(&ctrl->full[pending[0]]));
#pragma unroll
                for (int q = 0; q + 1 < kInFlight; ++q) pending[q] = pending[q + 1];
                --npending;
            }
            if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    // release what is still in flight, oldest first (also on the way out of
    // an abort: every copy this thread issued lands before it leaves)
    cp_async_wait_pending<0>();
    ptx::fence_proxy_async_smem();
    for (int q = 0; q < npending; ++q) ptx::mbar_arrive(ptx::smem_addr(&ctrl->full[pending[q]]));
}

template <int kKind, bool kTma, int kKpb>
__device__ __forceinline__ void run_mma(const Params &p, uint32_t smem_base, Ctrl *ctrl,
                                        uint32_t tmem_base, WaitCtl *wc)
{
    using T = Traits<kKind>;
    const int64_t num_tiles = p.tiles_m * p.tiles_n;
    const Sched sc = schedule(p);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    const uint32_t idesc = kTma ? idesc_with_n(T::kIdesc, p.bn) : T::kIdescKMajorB;
    // test hook: wait on a barrier nothing arrives at, so the wait runs out
    bool ok = !p.inject_stall || wait_bounded(ptx::smem_addr(&ctrl->never), 0, wc);
    for (int64_t t = sc.t0; ok && t < num_tiles; t += sc.dt) {
        if (!wait_bounded(ptx::smem_addr(&ctrl->tmem_empty[acc]), acc_phase ^ 1u, wc)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int64_t kb = sc.kb0; kb < sc.kb1; kb += kKpb) {
            if (!wait_bounded(ptx::smem_addr(&ctrl->full[stage]), phase, wc)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const bool second = kKpb == 2 && kb + 1 < sc.kb1;
#pragma unroll
            for (int h = 0; h < kKpb; ++h) {
                if (h == 1 && !second) break;
                const uint32_t sa = smem_base + stage * static_cast<uint32_t>(p.stage_bytes) +
                                    h * (A_TILE_BYTES + static_cast<uint32_t>(p.bn) * ROW_BYTES);
                const uint32_t sb = sa + A_TILE_BYTES;
#pragma unroll
                for (int k = 0; k < T::BK / T::UMMA_K; ++k) {
                    // A (K-major): advance 32 bytes along the swizzled row; 8-row
                    // groups of the tile are 1024 bytes apart.
                    const uint64_t da = ptx::smem_desc(sa + k * 32, 16, 1024, ptx::kSw128);
                    uint64_t db;
                    if constexpr (!T::kBNMajor || !kTma) {
                        // B staged K-major like A
                        db = ptx::smem_desc(sb + k * 32, 16, 1024, ptx::kSw128);
                    } else {
                        // B N-major: one MMA's K rows per step; boxes of 128
                        // bytes of columns are kNBoxBytes apart
                        db = ptx::smem_desc(sb + k * T::kNStep, T::kNBoxBytes, T::kNSbo, T::kNLayout);
                    }
                    ptx::umma<kKind>(d_tmem, da, db, idesc, (kb + h != sc.kb0 || k != 0) ? 1u : 0u);
                }
            }
            ptx::umma_commit(ptx::smem_addr(&ctrl->empty[stage]));
            if (++stage == static_cast<uint32_t>(p.stages)) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        ptx::umma_commit(ptx::smem_addr(&ctrl->tmem_full[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    // Every MMA this thread issued has finished before TMEM can be released.
    ptx::umma_commit(ptx::smem_addr(&ctrl->mma_done));
    drain_wait(ptx::smem_addr(&ctrl->mma_done), 0);
}

__device__ __forceinline__ float as_f(uint32_t u)
{
    return __uint_as_float(u);
}

// Store 32 consecutive accumulator columns of one row.
template <int kKind>
__device__ __forceinline__ void store_chunk(const Params &p, int64_t row, int64_t col,
                                            const uint32_t (&r)[32])
{
    using T = Traits<kKind>;
    if (row >= p.M) return;
    const float alpha = p.alpha, beta = p.beta;
    if constexpr (T::kElem == 2) {
        uint16_t *crow = reinterpret_cast<uint16_t *>(p.C) + row * p.ldc;
        if (p.vec_c && col + 31 < p.N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(crow + col) & 15u) == 0)) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 *dst = reinterpret_cast<uint4 *>(crow + col + q * 8);
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = alpha * as_f(r[q * 8 + e]);
                if (beta != 0.f) {
                    const uint4 old = *dst;
                    const uint32_t *w = reinterpret_cast<const uint32_t *>(&old);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack2<T::kBF>(w[e]);
                        v[2 * e] = fmaf(beta, f.x, v[2 * e]);
                        v[2 * e + 1] = fmaf(beta, f.y, v[2 * e + 1]);
                    }
                }
                *dst = make_uint4(pack2<T::kBF>(v[0], v[1]), pack2<T::kBF>(v[2], v[3]),
                                  pack2<T::kBF>(v[4], v[5]), pack2<T::kBF>(v[6], v[7]));
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (col + e < p.N) {
                    float v = alpha * as_f(r[e]);
                    if (beta != 0.f) v = fmaf(beta, load1<T::kBF>(crow + col + e), v);
                    crow[col + e] = round1<T::kBF>(v);
                }
            }
        }
    } else {
        float *crow = reinterpret_cast<float *>(p.C) + row * p.ldc;
        if (p.vec_c && col + 31 < p.N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(crow + col) & 15u) == 0)) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 *dst = reinterpret_cast<float4 *>(crow + col + q * 4);
                float4 v = make_float4(alpha * as_f(r[q * 4 + 0]), alpha * as_f(r[q * 4 + 1]),
                                       alpha * as_f(r[q * 4 + 2]), alpha * as_f(r[q * 4 + 3]));
                if (beta != 0.f) {
                    const float4 c = *dst;
                    v.x = fmaf(beta, c.x, v.x);
                    v.y = fmaf(beta, c.y, v.y);
                    v.z = fmaf(beta, c.z, v.z);
                    v.w = fmaf(beta, c.w, v.w);
                }
                *dst = v;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (col + e < p.N) {
                    float v = alpha * as_f(r[e]);
                    if (beta != 0.f) v = fmaf(beta, crow[col + e], v);
                    crow[col + e] = v;
                }
            }
        }
    }
}

// ---- epilogue through shared memory and TMA stores
//
// Each epilogue warp owns two 4 KB staging boxes of 32 rows x 128 bytes (64
// f16 or 32 f32 columns), written with the 128-byte swizzle (16-byte chunk j
// of row r at chunk position j ^ (r mod 8): the 8 rows a wavefront touches
// fall in distinct banks).  One lane stores a full box with a TMA tensor
// store, which writes whole lines and clips rows / columns outside C; the
// next box goes to the other buffer while the first is read out.
constexpr int EPI_BOX_BYTES = 4096;
constexpr int EPI_BYTES = 4 * 2 * EPI_BOX_BYTES;  // four warps, two boxes each

// Shared memory of the single-CTA kernel: stage ring, epilogue boxes,
// control block (plus slack to align the base to 1024 bytes).
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_BYTES + 1024 + static_cast<int>(sizeof(Ctrl));

template <int kKind>
constexpr int box_cols()
{
    return Traits<kKind>::kElem == 2 ? 64 : 32;
}

// C_old for one row and one box of columns (masked, zeros outside C).
template <int kKind>
__device__ __forceinline__ void load_old(const Params &p, int64_t row, int64_t col, float *old)
{
    constexpr int COLS = box_cols<kKind>();
#pragma unroll
    for (int e = 0; e < COLS; ++e) old[e] = 0.f;
    if (row >= p.M) return;
    if constexpr (Traits<kKind>::kElem == 2) {
        constexpr bool kBF = Traits<kKind>::kBF;
        const uint16_t *crow = reinterpret_cast<const uint16_t *>(p.C) + row * p.ldc;
        if (p.vec_c && col + COLS - 1 < p.N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(crow + col) & 15u) == 0)) {
#pragma unroll
            for (int q = 0; q < COLS / 8; ++q) {
                const uint4 u = *reinterpret_cast<const uint4 *>(crow + col + q * 8);
                const uint32_t *w = reinterpret_cast<const uint32_t *>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack2<kBF>(w[e]);
                    old[q * 8 + 2 * e] = f.x;
                    old[q * 8 + 2 * e + 1] = f.y;
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < COLS; ++e)
                if (col + e < p.N) old[e] = load1<kBF>(crow + col + e);
        }
    } else {
        const float *crow = reinterpret_cast<const float *>(p.C) + row * p.ldc;
        if (p.vec_c && col + COLS - 1 < p.N && DGEMM_CHECK((reinterpret_cast<uintptr_t>(crow + col) & 15u) == 0)) {
#pragma unroll
            for (int q = 0; q < COLS / 4; ++q) {
                const float4 f = *reinterpret_cast<const float4 *>(crow + col + q * 4);
                old[q * 4 + 0] = f.x;
                old[q * 4 + 1] = f.y;
                old[q * 4 + 2] = f.z;
                old[q * 4 + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < COLS; ++e)
                if (col + e < p.N) old[e] = crow[col + e];
        }
    }
}

// C whose base or pitch rules out 16-byte stores: the warp's 32 x 32 chunk
// (thread t holds row row0 + t) goes through shared memory and is stored row
// by row with one column per lane, so each store instruction writes one
// contiguous row segment instead of 32 rows.  Word e of row t sits at
// column e ^ t, so both the row-wise writes and the column-wise reads hit 32
// different banks.  Needs 32 x 32 x 4 bytes (one epilogue box) at `smem`.
static_assert(32 * 32 * 4 <= EPI_BOX_BYTES, "a warp's row-by-row staging fits one epilogue box");

template <int kKind>
__device__ __forceinline__ void store_chunk_by_rows(const Params &p, int64_t row0, int64_t col,
                                                    const uint32_t (&r)[32], uint32_t smem, int lane)
{
    using T = Traits<kKind>;
#pragma unroll
    for (int e = 0; e < 32; ++e)
        ptx::st_shared_b32(smem + (static_cast<uint32_t>(lane) * 32u + (static_cast<uint32_t>(e) ^ lane)) * 4u, r[e]);
    __syncwarp();
    const int64_t c = col + lane;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
        const int64_t row = row0 + i;
        if (row >= p.M || !DGEMM_CHECK(row >= 0)) break;  // warp-uniform
        const uint32_t u = ptx::ld_shared_b32(smem + (static_cast<uint32_t>(i) * 32u + (lane ^ static_cast<uint32_t>(i))) * 4u);
        if (c < p.N) {
            float v = p.alpha * __uint_as_float(u);
            if constexpr (T::kElem == 2) {
                uint16_t *dst = reinterpret_cast<uint16_t *>(p.C) + row * p.ldc + c;
                if (p.beta != 0.f) v = fmaf(p.beta, load1<T::kBF>(dst), v);
                *dst = round1<T::kBF>(v);
            } else {
                float *dst = reinterpret_cast<float *>(p.C) + row * p.ldc + c;
                if (p.beta != 0.f) v = fmaf(p.beta, *dst, v);
                *dst = v;
            }
        }
    }
    __syncwarp();  // the buffer is reused by the next chunk
}

// Drain one warp's 32 accumulator rows (TMEM address taddr, first row row0)
// x BN columns from n0 into C.  nbox counts the boxes this warp has stored;
// kBoxes staging boxes of EPI_BOX_BYTES at box_smem take turns (2: a box is
// filled while the previous one's store is still reading).  cols: columns to
// drain (p.bn by default).
template <int kKind, int kBoxes = 2>
__device__ __forceinline__ void drain_rows(const Params &p, const CUtensorMap *tmap_c,
                                           uint32_t taddr, int64_t row0, int64_t n0,
                                           uint32_t box_smem, int lane, uint32_t &nbox, int cols = 0)
{
    if (cols == 0) cols = p.bn;
    const int64_t row = row0 + lane;
    // the warp's TMEM columns lie inside the 512 allocated (warp-uniform)
    if (!DGEMM_CHECK((taddr & 0xFFFFu) + static_cast<uint32_t>(cols) <= static_cast<uint32_t>(TMEM_COLS))) return;
    if (!p.tma_store) {
#pragma unroll 1
        for (int c = 0; c < cols / 32; ++c) {
            uint32_t r[32];
            __syncwarp();  // tcgen05.ld is warp-collective (.sync.aligned)
            ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
            ptx::tmem_ld_wait();
            if (p.vec_c)
                store_chunk<kKind>(p, row, n0 + c * 32, r);
            else
                store_chunk_by_rows<kKind>(p, row0, n0 + c * 32, r, box_smem, lane);
        }
        return;
    }
    constexpr int COLS = box_cols<kKind>();
#pragma unroll 1
    for (int b = 0; b < cols / COLS; ++b) {
        const int64_t col0 = n0 + b * COLS;
        uint32_t r[COLS];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + b * COLS, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        if constexpr (COLS == 64)
            ptx::tmem_ld_32x32b_x32(taddr + b * COLS + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        ptx::tmem_ld_wait();
        if (row0 >= p.M || col0 >= p.N) continue;  // warp-uniform: nothing of C here
        float v[COLS];
#pragma unroll
        for (int e = 0; e < COLS; ++e) v[e] = p.alpha * __uint_as_float(r[e]);
        if (p.beta != 0.f) {
            float old[COLS];
            load_old<kKind>(p, row, col0, old);
#pragma unroll
            for (int e = 0; e < COLS; ++e) v[e] = fmaf(p.beta, old[e], v[e]);
        }
        const uint32_t buf = box_smem + (nbox % kBoxes) * EPI_BOX_BYTES;
        if (lane == 0 && nbox >= kBoxes) ptx::bulk_wait_read<kBoxes - 1>();  // this box's last store read it
        __syncwarp();
        const uint32_t rowbase = buf + static_cast<uint32_t>(lane) * 128u;
        if (!DGEMM_CHECK(lane < 32 && (nbox % kBoxes) < static_cast<uint32_t>(kBoxes))) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint4 q;
            if constexpr (Traits<kKind>::kElem == 2) {
                constexpr bool kBF = Traits<kKind>::kBF;
                q = make_uint4(pack2<kBF>(v[j * 8 + 0], v[j * 8 + 1]), pack2<kBF>(v[j * 8 + 2], v[j * 8 + 3]),
                               pack2<kBF>(v[j * 8 + 4], v[j * 8 + 5]), pack2<kBF>(v[j * 8 + 6], v[j * 8 + 7]));
            } else {
                q = make_uint4(__float_as_uint(v[j * 4 + 0]), __float_as_uint(v[j * 4 + 1]),
                               __float_as_uint(v[j * 4 + 2]), __float_as_uint(v[j * 4 + 3]));
            }
            ptx::st_shared_v4(rowbase + ((static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u)) << 4), q);
        }
        ptx::fence_proxy_async_smem();  // make the box visible to the TMA engine
        __syncwarp();
        // a TMA store starts at non-negative coordinates inside C
        if (lane == 0 && DGEMM_CHECK(row0 >= 0 && col0 >= 0 && row0 < p.M && col0 < p.N)) {
            ptx::tma_store_2d(tmap_c, buf, static_cast<int32_t>(col0), static_cast<int32_t>(row0));
            ptx::bulk_commit();
        }
        ++nbox;
    }
}

template <int kKind>
__device__ __forceinline__ void run_epilogue(const Params &p, const CUtensorMap *tmap_c, Ctrl *ctrl,
                                             uint32_t tmem_base, uint32_t epi_smem, int warp,
                                             int lane, WaitCtl *wc)
{
    const int64_t num_tiles = p.tiles_m * p.tiles_n;
    const Sched sc = schedule(p);
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);  // TMEM lanes this warp may read
    uint32_t acc = 0, acc_phase = 0, nbox = 0;
    for (int64_t t = sc.t0; t < num_tiles; t += sc.dt) {
        int64_t m0, n0;
        tile_coords(t, p, m0, n0);
        bool ok = wait_bounded(ptx::smem_addr(&ctrl->tmem_full[acc]), acc_phase, wc);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + ((quarter * 32u) << 16) + acc * BN;
        // the schedule's tile lies inside C (warp-uniform)
        if (DGEMM_CHECK(m0 >= 0 && m0 < p.M && n0 >= 0 && n0 < p.N))
            drain_rows<kKind>(p, tmap_c, taddr, m0 + quarter * 32, n0,
                              epi_smem + quarter * 2 * EPI_BOX_BYTES, lane, nbox);
        ptx::tc_fence_before();
        ptx::mbar_arrive(ptx::smem_addr(&ctrl->tmem_empty[acc]));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait<0>();  // stores done before the CTA leaves
}

// ---- split-K: the partial sums of a tile meet in distributed shared memory
//
// Each of the S CTAs of a cluster has summed its K range of the same tile in
// TMEM.  The tile's eight 32-column chunks are owned round-robin: chunk c by
// rank c mod S.  A first cluster barrier, reached by each CTA's epilogue
// warps only after its accumulator is complete, guarantees that no CTA still
// reads or fills its stage ring.  "push": every CTA then copies the chunks it
// does not own from TMEM straight into the owner's idle stage buffers --
// remote 16-byte stores, which the thread does not wait for.  After a second
// cluster barrier,
// "reduce": the owner adds, for each row and column, the S partials in rank
// order 0..S-1 (its own taken from TMEM, the others from its shared memory),
// so the sum does not depend on timing, and stores alpha * sum + beta * C_old.
// Nothing crosses CTAs after that barrier, so each CTA leaves when its own
// reduction is done.
// Layout of the receive buffers, in 16-byte units: [slot = sender among the
// other S-1 ranks][owned chunk][column quad q][row]; consecutive threads
// (rows) touch consecutive 16-byte words, so a warp moves 512 contiguous
// bytes per access.

constexpr uint32_t splitk_recv_bytes(uint32_t S)
{
    return (S - 1) * ((BN / 32 + S - 1) / S) * 8u * BM * 16u;
}
static_assert(splitk_recv_bytes(2) <= STAGES * STAGE_BYTES && splitk_recv_bytes(3) <= STAGES * STAGE_BYTES &&
                  splitk_recv_bytes(4) <= STAGES * STAGE_BYTES && splitk_recv_bytes(5) <= STAGES * STAGE_BYTES &&
                  splitk_recv_bytes(6) <= STAGES * STAGE_BYTES && splitk_recv_bytes(7) <= STAGES * STAGE_BYTES &&
                  splitk_recv_bytes(8) <= STAGES * STAGE_BYTES,
              "split-K partials must fit in the stage ring");

__device__ __forceinline__ uint32_t recv_offset(uint32_t slot, uint32_t chunk_idx, uint32_t S,
                                                int q, int row)
{
    const uint32_t owned_max = (BN / 32 + S - 1) / S;
    return (((slot * owned_max + chunk_idx) * 8u + static_cast<uint32_t>(q)) * BM +
            static_cast<uint32_t>(row)) * 16u;
}

// The accumulator of this CTA's K range is complete (its MMAs, and with them
// every read of its stage ring, are done).  Bounded; a time-out raises the
// CTA's abort flag, which push and reduce check.
__device__ __forceinline__ void splitk_wait_acc(Ctrl *ctrl, WaitCtl *wc)
{
    wait_bounded(ptx::smem_addr(&ctrl->tmem_full[0]), 0, wc);
}

__device__ __forceinline__ void splitk_push(const Params &p, uint32_t tmem_base, uint32_t smem_base,
                                            int warp, int lane, WaitCtl *wc)
{
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    if (__any_sync(0xffffffffu, aborted(wc))) return;
    ptx::tc_fence_after();
    const uint32_t S = static_cast<uint32_t>(p.splitk);
    const uint32_t rank = ptx::cluster_ctarank();
    const int row = static_cast<int>(quarter * 32 + lane);
    const uint32_t taddr = tmem_base + ((quarter * 32u) << 16);
#pragma unroll 1
    for (int c = 0; c < p.bn / 32; ++c) {
        const uint32_t owner = static_cast<uint32_t>(c) % S;
        if (owner == rank) continue;
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
        ptx::tmem_ld_wait();
        const uint32_t slot = rank < owner ? rank : rank - 1;
        // the eight 16-byte words land inside the owner's stage ring
        if (!DGEMM_CHECK(owner < S && recv_offset(slot, static_cast<uint32_t>(c) / S, S, 7, row) + 16 <=
                                          static_cast<uint32_t>(STAGES * STAGE_BYTES)))
            continue;
        const uint32_t base = ptx::mapa(smem_base + recv_offset(slot, static_cast<uint32_t>(c) / S, S, 0, row),
                                        owner);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ptx::st_shared_cluster_v4(base + static_cast<uint32_t>(q) * BM * 16u,
                                      make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                  __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
    }
}

template <int kKind>
__device__ __forceinline__ void splitk_reduce(const Params &p, uint32_t tmem_base,
                                              uint32_t smem_base, int warp, int lane, WaitCtl *wc)
{
    if (__any_sync(0xffffffffu, aborted(wc))) return;
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    const uint32_t S = static_cast<uint32_t>(p.splitk);
    const uint32_t rank = ptx::cluster_ctarank();
    int64_t m0, n0;
    tile_coords(blockIdx.x / S, p, m0, n0);
    const int row = static_cast<int>(quarter * 32 + lane);
    const uint32_t taddr = tmem_base + ((quarter * 32u) << 16);
    ptx::tc_fence_after();
#pragma unroll 1
    for (uint32_t c = rank; c < static_cast<uint32_t>(p.bn) / 32; c += S) {
        uint32_t own[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, own);
        ptx::tmem_ld_wait();
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
        for (uint32_t q = 0; q < S; ++q) {
            if (q == rank) {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] += __uint_as_float(own[j]);
            } else {
                const uint32_t slot = q < rank ? q : q - 1;
                const uint32_t base = smem_base + recv_offset(slot, c / S, S, 0, row);
                if (!DGEMM_CHECK(recv_offset(slot, c / S, S, 7, row) + 16 <= static_cast<uint32_t>(STAGES * STAGE_BYTES)))
                    continue;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const float4 f = ptx::ld_shared_v4f(base + static_cast<uint32_t>(v) * BM * 16u);
                    acc[4 * v] += f.x;
                    acc[4 * v + 1] += f.y;
                    acc[4 * v + 2] += f.z;
                    acc[4 * v + 3] += f.w;
                }
            }
        }
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
        store_chunk<kKind>(p, m0 + row, n0 + c * 32, r);
    }
}

// Threads per CTA: producer warp(s), one MMA warp, four epilogue warps.
template <bool kTma>
constexpr int producer_warps()
{
    return kTma ? 1 : 4;
}
template <bool kTma>
constexpr int cta_threads()
{
    return 32 * (producer_warps<kTma>() + 1 + 4);
}

// kKpb: K blocks per stage of the TMA producer (p.kpb; 1 for the non-TMA
// producers).  Two instances rather than a run-time count: the one-block
// kernel keeps the code (and the cold-start instruction fetches) of a
// single block per stage.
template <int kKind, bool kTma, int kKpb = 1>
__global__ void __launch_bounds__(cta_threads<kTma>(), 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, const Params p)
{
    constexpr int kMmaWarp = producer_warps<kTma>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctrl->full[s]), kTma ? 1 : 32 * producer_warps<kTma>());
            ptx::mbar_init(ptx::smem_addr(&ctrl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&ctrl->tmem_full[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctrl->tmem_empty[a]), 4 * 32);
        }
        ptx::mbar_init(ptx::smem_addr(&ctrl->mma_done), 1);
        ptx::mbar_init(ptx::smem_addr(&ctrl->never), 1);
        ctrl->wait.abort = 0;
        ctrl->wait.limit_ns = p.wait_limit_ns;
        ptx::fence_mbarrier_init();
    }
    if (kTma && warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
    }
    if (p.tma_store && warp == kMmaWarp + 1 && lane == 0) ptx::prefetch_tmap(&tmap_c);
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&ctrl->tmem_base), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl->tmem_base;
    WaitCtl *wc = &ctrl->wait;
    const uint32_t smem_base = ptx::smem_addr(smem);

    if (warp < kMmaWarp) {
        if constexpr (kTma) {
            if (lane == 0) run_producer<kKind, kKpb>(&tmap_a, &tmap_b, p, smem_base, ctrl, wc);
        } else if constexpr (kKind == kTF32) {
            run_cpasync_producer(p, smem_base, ctrl, threadIdx.x, wc);
        } else {
            run_reg_producer<kKind>(p, smem_base, ctrl, threadIdx.x, wc);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) run_mma<kKind, kTma, kKpb>(p, smem_base, ctrl, tmem_base, wc);
    } else {
        if (p.splitk > 1)
            splitk_wait_acc(ctrl, wc);
        else
            run_epilogue<kKind>(p, &tmap_c, ctrl, tmem_base, smem_base + STAGES * STAGE_BYTES, warp,
                                lane, wc);
    }

    if (p.splitk > 1) {  // uniform over the cluster
        __syncwarp();
        ptx::tc_fence_before();
        ptx::cluster_sync();  // every CTA's accumulator is complete: all stage rings are idle
        if (warp > kMmaWarp) splitk_push(p, tmem_base, smem_base, warp, lane, wc);
        __syncwarp();
        ptx::tc_fence_before();
        ptx::cluster_sync();  // every pushed partial has landed in its owner
        if (warp > kMmaWarp) splitk_reduce<kKind>(p, tmem_base, smem_base, warp, lane, wc);
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA pairs
//
// The same GEMM on a pair of CTAs (a cluster of 2 on neighbouring SMs) that
// share one tcgen05.mma of 256 x 256 x UMMA_K (cta_group::2): each CTA loads
// its own 128 rows of A and one half (128 columns) of B, and holds its 128
// rows of the 256 x 256 accumulator in its own TMEM.  Per CTA the operand
// bytes per output tile fall from (128 + 256) to (128 + 128) rows per K slice,
// which is what bounds the single-CTA kernel (L2 -> SM bandwidth).
//   both CTAs  warp 0: TMA producer into the CTA's own 6-stage ring; both
//              CTAs' loads complete on the even CTA's "full" barrier, which
//              the even producer arms with the bytes of both halves;
//              warps 2-5: epilogue of the CTA's 128 rows;
//   even CTA   warp 6: waits for each stage's "full" barrier and hands the
//              stage to warp 1 through a named CTA barrier;
//              warp 1: the MMA issuer for the pair (one lane issues); it
//              multicasts its commits to both CTAs' "empty" / "tmem_full"
//              barriers.
// The epilogue warps of both CTAs release an accumulator by arriving on the
// even CTA's "tmem_empty" barrier (8 warp arrivals).
//
// Why a separate waiter: measured on GB300, an mbarrier probe (or any
// shared-memory access) that the MMA-issuing thread makes between one
// stage's MMAs and the next costs ~25 % of tensor throughput at 256 x 256
// tiles -- the thread cannot issue the next stage until the probe returns,
// and the tensor pipe runs dry meanwhile.  A named barrier (bar.red) does not
// have that cost: with the waits moved to warp 6, the MMA warp keeps the pipe
// at ~97 % of its peak when the operands are already in shared memory.

constexpr int PAIR_STAGES = 6;
constexpr int PAIR_MAX_STAGES = 12;                // the finer ring (see PairShape)
constexpr int PAIR_BM = 2 * BM;                    // rows per pair tile
constexpr int PAIR_HALF_BYTES = 128 * ROW_BYTES;   // 16 KB: 128 rows of A or of B
constexpr int PAIR_STAGE_BYTES = 2 * PAIR_HALF_BYTES;
constexpr int PAIR_THREADS = 224;
// Wide tiles (kWide = 2) drain a 512-column accumulator that the next tile's
// MMAs wait for, so they add four epilogue warps (7-10): each of the eight
// drains one lane quarter x 256 columns, with one staging box each.
template <int kWide>
constexpr int pair_threads()
{
    return kWide == 2 ? PAIR_THREADS + 4 * 32 : PAIR_THREADS;
}
constexpr int PAIR_MMA_WARP = 1;
constexpr int PAIR_WAITER_WARP = 6;
constexpr uint32_t PAIR_HANDOFF_THREADS = 64;  // warps 1 and 6 on named barriers 1..stages

struct PairCtrl {
    uint64_t full[PAIR_MAX_STAGES];   // even CTA: both halves of the stage landed
    uint64_t empty[PAIR_MAX_STAGES];  // the pair's MMAs have read this stage
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t acc_ready;  // stream-K: every epilogue warp has loaded its part of a partial
    uint64_t mma_done;
    uint64_t never;  // test hook: a barrier nothing arrives at
    WaitCtl wait;
    uint32_t tmem_base;
};

constexpr int PAIR_SMEM_BYTES =
    PAIR_STAGES * PAIR_STAGE_BYTES + EPI_BYTES + 1024 + static_cast<int>(sizeof(PairCtrl));

template <int kKind>
constexpr uint32_t pair_idesc()
{
    return (Traits<kKind>::kIdesc & ~(0x1Fu << 24)) | (static_cast<uint32_t>(PAIR_BM >> 4) << 24);
}

// Output tile of pair tile t: 256 rows from m0, p.bn columns from n0.
__device__ __forceinline__ void pair_tile(int64_t t, const Params &p, int64_t &m0, int64_t &n0)
{
    tile_coords(t, p, m0, n0, PAIR_BM);
}

// Pair tiles of 256 x (256 * kWide): with kWide = 2 each MMA step is two
// MMAs of N = 256 into one 512-column accumulator (the whole TMEM), so each
// CTA loads 16 KB of A and 32 KB of B per stage for twice the MMA work --
// a quarter fewer bytes per flop into every SM -- at the price of a single
// accumulator, whose drain the next tile's MMAs wait for.
//
// kRowB is the K depth of a stage in bytes per row: 128 (one 128-byte
// swizzled row: 64 f16 / 32 f32 elements), or 64 -- the finer ring of the
// K-major 16-bit kinds: rows of 32 elements under the 64-byte swizzle, so a
// stage is half as large, the same 192 KB hold twice as many, and the MMAs
// release their stage after two instructions instead of four.
template <int kWide, int kRowB = ROW_BYTES>
struct PairShape {
    static constexpr int kHalfBytes = 128 * kRowB;                      // 128 rows of A or of B
    static constexpr int kStageBytes = kHalfBytes * (1 + kWide);        // A half + kWide B halves
    static constexpr int kStages = PAIR_STAGES * PAIR_STAGE_BYTES / kStageBytes;  // 6 / 4, or 12 / 8
    static constexpr int kAccs = 2 / kWide;                             // TMEM accumulators
    static constexpr int kAccCols = BN * kWide;
    static constexpr uint32_t kSbo = 8u * kRowB;                        // bytes between 8-row groups
    static constexpr uint32_t kLayout = kRowB == ROW_BYTES ? ptx::kSw128 : ptx::kSw64;
    static_assert(kRowB == ROW_BYTES || kRowB == 64, "stages of 128 or 64 bytes of K per row");
    static_assert(kStages <= PAIR_MAX_STAGES, "barriers for every stage");
    static_assert(kStageBytes % 1024 == 0, "stages start on the swizzle pattern's period");
};

// ---- stream-K tail
//
// With T tiles on P pairs and T mod P = r != 0, whole tiles dealt round-robin
// leave r pairs busy in the last round and P - r idle.  Instead the first
// P + r tiles of the tile order are cut along K: their (P + r) x num_kb K
// blocks are dealt in P contiguous ranges, one per pair (at least num_kb
// blocks each, so no range lies strictly inside one tile and each tile is
// cut at most once); the remaining (T / P - 1) x P tiles go round-robin.
// A pair walks its range from its last tile back to its first:
//   * the head [0, k) of its last tile (when the range ends inside it) comes
//     first; its raw f32 accumulator goes to the pair's slot of sk_work
//     ("publish") and each epilogue warp stamps its flag with sk_gen;
//   * whole tiles in between are ordinary;
//   * the tail [k, num_kb) of its first tile comes last: each epilogue warp
//     waits for the previous pair's flag, loads that partial into TMEM
//     ("init"), and the MMAs accumulate onto it.
// The MMAs of a cut tile therefore run in exactly the order of an uncut one,
// so the result is bit-identical to the round-robin schedule.  A partial is
// published at the start of a pair's work and consumed at the end of the
// next pair's, so the wait is normally already satisfied.
struct Unit {
    int64_t t;       // tile in tile order
    int64_t k0, k1;  // K blocks [k0, k1)
    bool init;       // start from the previous pair's partial (k0 > 0)
    bool publish;    // leave the partial for the next pair (k1 < num_kb)
};

struct WorkIter {
    int64_t t_sk, t_sk_first, b, e;  // stream-K: next tile (descending), first tile, K-block range
    int64_t t_dp, dt_dp, tiles;      // round-robin: next tile, stride, tile count

    __host__ __device__ __forceinline__ WorkIter(const Params &p, int64_t cluster, int64_t clusters)
    {
        tiles = p.tiles_m * p.tiles_n;
        if (p.sk_tiles > 0) {
            const int64_t blocks = p.sk_tiles * p.num_kb;
            b = cluster * blocks / clusters;
            e = (cluster + 1) * blocks / clusters;
            t_sk_first = b / p.num_kb;
            t_sk = (e - 1) / p.num_kb;
        } else {
            b = e = 0;
            t_sk_first = 0;
            t_sk = -1;
        }
        t_dp = p.sk_tiles + cluster;
        dt_dp = clusters;
    }

    // whether the unit after the current one is the "init" tail
    __host__ __device__ __forceinline__ bool next_is_init(const Params &p) const
    {
        return t_sk == t_sk_first && b > t_sk_first * p.num_kb;
    }

    __host__ __device__ __forceinline__ bool next(const Params &p, Unit &u)
    {
        if (t_sk >= t_sk_first) {
            const int64_t base = t_sk * p.num_kb;
            u.t = t_sk;
            u.k0 = b > base ? b - base : 0;
            u.k1 = e < base + p.num_kb ? e - base : p.num_kb;
            u.init = u.k0 > 0;
            u.publish = u.k1 < p.num_kb;
            --t_sk;
            return true;
        }
        if (t_dp < tiles) {
            u.t = t_dp;
            u.k0 = 0;
            u.k1 = p.num_kb;
            u.init = u.publish = false;
            t_dp += dt_dp;
            return true;
        }
        return false;
    }
};

// Partials: per pair slot, CTA half and epilogue warp (8 slots; the 256-wide
// tiles use 4) a region of 32 rows x 256 columns of f32 = 32 KB, laid out
// [32-column chunk][column quad][row] in 16-byte units so that each warp
// access is 512 contiguous bytes.  One flag per region.
constexpr int SK_WARP_SLOTS = 8;
constexpr int64_t SK_REGION_FLOATS = 32 * 256;
constexpr int SK_MAX_PAIRS = 128;  // pair slots of the static workspace
constexpr int64_t SK_REGIONS = static_cast<int64_t>(SK_MAX_PAIRS) * 2 * SK_WARP_SLOTS;

__device__ __forceinline__ int64_t sk_region(int64_t slot, uint32_t half, int w)
{
    return (slot * 2 + half) * SK_WARP_SLOTS + w;
}

// Store this warp's 32 rows x cols accumulator columns (cols a multiple of 32)
// to its region.  The caller may release TMEM afterwards, then stamps the
// flag with sk_flag().
__device__ __forceinline__ void sk_publish(const Params &p, uint32_t taddr, int cols, int64_t region,
                                          int lane)
{
    if (!DGEMM_CHECK(region >= 0 && region < SK_REGIONS && cols <= 256)) return;  // warp-uniform
    float4 *dst = reinterpret_cast<float4 *>(p.sk_work + region * SK_REGION_FLOATS);
#pragma unroll 1
    for (int c = 0; c < cols / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(taddr + c * 32, r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[(c * 8 + j) * 32 + lane] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                       __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    }
}

// Stamp the region's flag once every lane's stores are visible (release).
__device__ __forceinline__ void sk_flag(const Params &p, int64_t region, int lane)
{
    if (!DGEMM_CHECK(region >= 0 && region < SK_REGIONS)) return;  // warp-uniform
    __threadfence();
    __syncwarp();
    if (lane == 0) ptx::st_release_gpu_u64(p.sk_flags + region, p.sk_gen);
}

// If the region's partial is already published, pull its lines into L2 (the
// warp is otherwise idle, waiting for an accumulator), so that sk_init's
// loads do not go to HBM.
__device__ __forceinline__ void sk_prefetch(const Params &p, int cols, int64_t region, int lane)
{
    if (!DGEMM_CHECK(region >= 0 && region < SK_REGIONS)) return;
    const bool ready = ptx::ld_acquire_gpu_u64(p.sk_flags + region) == p.sk_gen;
    if (!ready) return;
    const char *base = reinterpret_cast<const char *>(p.sk_work + region * SK_REGION_FLOATS);
    const int lines = cols * 32 * 4 / 128;  // 128-byte lines of the region in use
    for (int l = lane; l < lines; l += 32) ptx::prefetch_l2(base + static_cast<int64_t>(l) * 128);
}

// Wait (bounded) for the region's flag to carry this launch's generation,
// then load the partial into this warp's 32 TMEM lanes x BN columns, two
// chunks in flight.  False on time-out or abort.
__device__ __forceinline__ bool sk_init(const Params &p, uint32_t taddr, int64_t region, int lane, WaitCtl *wc)
{
    constexpr int kChunks = BN / 32;
    static_assert(kChunks % 2 == 0, "chunks are loaded in pairs");
    // a region of the workspace, and TMEM columns inside the allocation (warp-uniform)
    if (!DGEMM_CHECK(region >= 0 && region < SK_REGIONS && (taddr & 0xFFFFu) + BN <= static_cast<uint32_t>(TMEM_COLS)))
        return false;
    bool ok = true;
    if (lane == 0) {
        const uint64_t *flag = p.sk_flags + region;
        if (ptx::ld_acquire_gpu_u64(flag) != p.sk_gen) {
            const uint64_t t0 = ptx::globaltimer_ns();
            for (;;) {
                if (ptx::ld_acquire_gpu_u64(flag) == p.sk_gen) break;
                if (aborted(wc)) {
                    ok = false;
                    break;
                }
                if (ptx::globaltimer_ns() - t0 > wc->limit_ns) {
                    raise_abort(wc);
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
        }
    }
    if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) return false;
    (void)ptx::ld_acquire_gpu_u64(p.sk_flags + region);  // every lane acquires before its loads
    const uint4 *src = reinterpret_cast<const uint4 *>(p.sk_work + region * SK_REGION_FLOATS) + lane;
    // chunks c and c + 1 in two register sets (L2 loads: written during this launch)
    uint32_t ra[32], rb[32];
    auto load = [&](uint32_t (&r)[32], int c) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 v = __ldcg(src + (c * 8 + j) * 32);
            r[4 * j] = v.x;
            r[4 * j + 1] = v.y;
            r[4 * j + 2] = v.z;
            r[4 * j + 3] = v.w;
        }
    };
    load(ra, 0);
#pragma unroll 1
    for (int c = 0; c < kChunks; c += 2) {
        load(rb, c + 1);
        ptx::tmem_st_32x32b_x32(taddr + c * 32, ra);
        if (c + 2 < kChunks) load(ra, c + 2);
        ptx::tmem_st_32x32b_x32(taddr + (c + 1) * 32, rb);
    }
    ptx::tmem_st_wait();
    return true;
}

template <int kKind, int kWide, int kRowB>
__device__ __forceinline__ void pair_producer(const CUtensorMap *tmap_a, const CUtensorMap *tmap_b,
                                              const CUtensorMap *tmap_b2, const Params &p, uint32_t smem_base,
                                              PairCtrl *ctrl, uint32_t rank, WaitCtl *wc)
{
    using T = Traits<kKind>;
    using S = PairShape<kWide, kRowB>;
    constexpr int kStageK = kRowB / T::kElem;  // K elements per stage
    const int64_t cluster = blockIdx.x / 2, clusters = gridDim.x / 2;
    const uint32_t half = rank & 1u;
    uint32_t stage = 0, phase = 0;
    uint32_t issued = 0, issued_phase = 0;
    bool ok = true;
    WorkIter it(p, cluster, clusters);
    Unit u;
    while (ok && it.next(p, u)) {
        int64_t m0, n0;
        pair_tile(u.t, p, m0, n0);
        for (int64_t kb = u.k0; kb < u.k1; ++kb) {
            if (!wait_bounded_cluster(ptx::smem_addr(&ctrl->empty[stage]), phase ^ 1u, wc)) {
                ok = false;
                break;
            }
            const uint32_t full_local = ptx::smem_addr(&ctrl->full[stage]);
            const uint32_t full = ptx::mapa(full_local, 0);  // the pair leader's barrier
            if (half == 0) ptx::mbar_arrive_expect_tx(full_local, 2 * S::kStageBytes);
            const uint32_t sa = smem_base + stage * S::kStageBytes;
            const int32_t kc = static_cast<int32_t>(kb * kStageK);
            ptx::tma_load_2d_pair(sa, tmap_a, full, kc, static_cast<int32_t>(m0 + half * 128));
#pragma unroll
            for (int w = 0; w < kWide; ++w) {
                const uint32_t sb = sa + (1 + w) * S::kHalfBytes;
                const int64_t nb = n0 + w * BN + half * 128;  // this CTA's half of B, MMA w
                if constexpr (!T::kBNMajor) {
                    ptx::tma_load_2d_pair(sb, tmap_b, full, kc, static_cast<int32_t>(nb));
                } else if (p.b3d && nb + 128 <= p.b3d_cols) {
                    // one instruction instead of four (TF32) or two (16-bit NN):
                    // the producer thread's issue rate bounds the TF32 stage rate
                    ptx::tma_load_3d_pair(sb, tmap_b, full, 0, kc, static_cast<int32_t>(nb / T::kNBox));
                } else {
                    // 2-D boxes of one column group each (zeros past N)
                    const CUtensorMap *m2 = p.b3d ? tmap_b2 : tmap_b;
#pragma unroll
                    for (int c = 0; c < 128 / T::kNBox; ++c)
                        ptx::tma_load_2d_pair(sb + c * T::kNBoxBytes, m2, full,
                                              static_cast<int32_t>(nb + c * T::kNBox), kc);
                }
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == S::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok && half == 0) {
        // The leader's barrier counts both CTAs' bytes: wait (bounded) for
        // the loads in flight before the pair leaves.
        for (int s = 0; s < S::kStages; ++s)
            if ((issued >> s) & 1u)
                drain_wait(ptx::smem_addr(&ctrl->full[s]), (issued_phase >> s) & 1u);
    }
}

// A pair leader's full-barrier waiter (warp 6): for every stage the pair
// consumes, waits (bounded) for its "full" barrier, then meets the MMA warp on
// named barrier 1 + stage.  The barrier's OR-reduction carries the abort flag
// both ways, so each side runs through the same number of hand-offs and
// neither can be left waiting on the other after a time-out.
template <int kKind, int kWide, int kRowB>
__device__ __forceinline__ void pair_waiter(const Params &p, PairCtrl *ctrl, int lane, WaitCtl *wc)
{
    using S = PairShape<kWide, kRowB>;
    const int64_t cluster = blockIdx.x / 2, clusters = gridDim.x / 2;
    uint32_t stage = 0, phase = 0;
    bool abort = false;
    WorkIter it(p, cluster, clusters);
    Unit u;
    while (it.next(p, u)) {
        for (int64_t kb = u.k0; kb < u.k1; ++kb) {
            if (!abort) {
                bool ok = true;
                if (lane == 0) ok = wait_bounded_cluster(ptx::smem_addr(&ctrl->full[stage]), phase, wc);
                abort = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0) != 0;
            }
            abort = ptx::bar_red_or(1 + stage, PAIR_HANDOFF_THREADS, abort);
            if (++stage == S::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// A pair's MMA warp (warp 1 of the leader; lane 0 issues).  Per stage it
// takes the hand-off from the waiter, issues the stage's MMAs and commits the
// stage's release to the "empty" barriers of both CTAs; per tile it waits
// for a free accumulator and commits "tmem_full" to both CTAs.
template <int kKind, int kWide, int kRowB>
__device__ __forceinline__ void pair_mma(const Params &p, uint32_t smem_base, PairCtrl *ctrl,
                                         uint32_t tmem_base, uint32_t rank, int lane, WaitCtl *wc)
{
    using T = Traits<kKind>;
    using S = PairShape<kWide, kRowB>;
    constexpr int kStageK = kRowB / T::kElem;  // K elements per stage
    constexpr uint16_t kBoth = 0x3;  // the two CTAs of the pair
    const int64_t cluster = blockIdx.x / 2, clusters = gridDim.x / 2;
    uint32_t stage = 0, acc = 0, acc_phase = 0, ready_phase = 0;
    // test hook: wait on a barrier nothing arrives at, so the wait runs out
    bool ok = true;
    if (lane == 0 && p.inject_stall) ok = wait_bounded(ptx::smem_addr(&ctrl->never), 0, wc);
    bool abort = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0) != 0;
    WorkIter it(p, cluster, clusters);
    Unit u;
    while (it.next(p, u)) {
        if (!abort) {
            ok = true;
            if (lane == 0)
                ok = wait_bounded_cluster(ptx::smem_addr(&ctrl->tmem_empty[acc]), acc_phase ^ 1u, wc);
            // stream-K: the epilogue warps load the previous pair's partial first
            if (ok && lane == 0 && u.init) ok = wait_bounded_cluster(ptx::smem_addr(&ctrl->acc_ready), ready_phase, wc);
            abort = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0) != 0;
        }
        if (u.init) ready_phase ^= 1u;
        const uint32_t acc_first = u.init ? 1u : 0u;  // accumulate onto the loaded partial
        const uint32_t d_tmem = tmem_base + acc * S::kAccCols;
        for (int64_t kb = u.k0; kb < u.k1; ++kb) {
            abort = ptx::bar_red_or(1 + stage, PAIR_HANDOFF_THREADS, abort);
            if (!abort) {
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = smem_base + stage * S::kStageBytes;
#pragma unroll
                    for (int k = 0; k < kStageK / T::UMMA_K; ++k) {
                        // K-major: advance 32 bytes along the swizzled row; 8-row
                        // groups are 8 rows of kRowB bytes apart
                        const uint64_t da = ptx::smem_desc(sa + k * 32, 16, S::kSbo, S::kLayout);
#pragma unroll
                        for (int w = 0; w < kWide; ++w) {
                            const uint32_t sb = sa + (1 + w) * S::kHalfBytes;
                            uint64_t db;
                            if constexpr (!T::kBNMajor)
                                db = ptx::smem_desc(sb + k * 32, 16, S::kSbo, S::kLayout);
                            else
                                db = ptx::smem_desc(sb + k * T::kNStep, T::kNBoxBytes, T::kNSbo, T::kNLayout);
                            ptx::umma_pair<kKind>(d_tmem + w * BN, da, db, pair_idesc<kKind>(),
                                                  (kb != u.k0 || k != 0) ? 1u : acc_first);
                        }
                    }
                    ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->empty[stage]), kBoth);
                }
                __syncwarp();
            }
            if (++stage == S::kStages) stage = 0;
        }
        if (!abort && lane == 0) ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->tmem_full[acc]), kBoth);
        __syncwarp();
        if (++acc == S::kAccs) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    if (lane == 0) {
        ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->mma_done), static_cast<uint16_t>(1u << rank));
        drain_wait(ptx::smem_addr(&ctrl->mma_done), 0);
    }
    __syncwarp();
}

template <int kKind, int kWide>
__device__ __forceinline__ void pair_epilogue(const Params &p, const CUtensorMap *tmap_c,
                                              PairCtrl *ctrl, uint32_t tmem_base, uint32_t epi_smem,
                                              uint32_t rank, int warp, int lane, WaitCtl *wc)
{
    const int64_t cluster = blockIdx.x / 2, clusters = gridDim.x / 2;
    const uint32_t quarter = static_cast<uint32_t>(warp & 3);
    const uint32_t leader = rank & ~1u;
    // kWide = 2: warps 2-5 drain columns 0-255, warps 7-10 columns 256-511
    const uint32_t colhalf = kWide == 2 && warp >= 7 ? 1u : 0u;
    const int slot = kWide == 2 ? warp - (warp >= 7 ? 3 : 2) : warp - 2;  // 0..7 / 0..3
    const uint32_t box = kWide == 2 ? epi_smem + static_cast<uint32_t>(slot) * EPI_BOX_BYTES
                                    : epi_smem + quarter * 2 * EPI_BOX_BYTES;
    constexpr int kAccs = PairShape<kWide>::kAccs;
    uint32_t acc = 0, acc_phase = 0, nbox = 0;
    WorkIter it(p, cluster, clusters);
    Unit u;
    while (it.next(p, u)) {
        int64_t m0, n0;
        pair_tile(u.t, p, m0, n0);
        const uint32_t taddr = tmem_base + ((quarter * 32u) << 16) + acc * PairShape<kWide>::kAccCols +
                               colhalf * BN;
        // Stream-K "init": load the previous pair's partial into the unit's
        // accumulator before its MMAs.  With two accumulators it is done one
        // unit ahead, while this unit's MMAs run: the next unit's accumulator
        // was drained in the previous iteration.  With one, it waits for this
        // unit (the accumulator is free only now); the lines are pulled into
        // L2 a unit ahead instead.
        bool init_now = kAccs == 1 && u.init;
        uint32_t init_addr = taddr;
        if (kAccs == 2 && it.next_is_init(p)) {
            init_now = true;
            init_addr = acc ? taddr - PairShape<kWide>::kAccCols : taddr + PairShape<kWide>::kAccCols;  // the other one
        } else if (kAccs == 1 && it.next_is_init(p)) {
            sk_prefetch(p, BN, sk_region(cluster - 1, rank & 1u, slot), lane);
        }
        if (init_now) {
            if (!sk_init(p, init_addr, sk_region(cluster - 1, rank & 1u, slot), lane, wc)) break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_addr(&ctrl->acc_ready), leader));
        }
        bool ok = wait_bounded_cluster(ptx::smem_addr(&ctrl->tmem_full[acc]), acc_phase, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ptx::tc_fence_after();
        if (!DGEMM_CHECK(m0 >= 0 && m0 < p.M && n0 >= 0 && n0 < p.N && static_cast<uint32_t>(slot) < 8u)) {
            // (the schedule's tile lies inside C; nothing is drained otherwise)
        } else if (u.publish)
            sk_publish(p, taddr, BN, sk_region(cluster, rank & 1u, slot), lane);
        else if constexpr (kWide == 2)
            drain_rows<kKind, 1>(p, tmap_c, taddr, m0 + (rank & 1u) * 128 + quarter * 32,
                                 n0 + colhalf * BN, box, lane, nbox, BN);
        else
            drain_rows<kKind>(p, tmap_c, taddr, m0 + (rank & 1u) * 128 + quarter * 32, n0, box, lane, nbox);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)
            ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_addr(&ctrl->tmem_empty[acc]), leader));
        if (u.publish) sk_flag(p, sk_region(cluster, rank & 1u, slot), lane);  // after TMEM is released
        if (++acc == PairShape<kWide>::kAccs) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    if (lane == 0) ptx::bulk_wait<0>();  // stores done before the CTA leaves
}

template <int kKind, int kWide, int kRowB = ROW_BYTES>
__global__ void __launch_bounds__(pair_threads<kWide>(), 1)
    umma_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_b2,
                     const __grid_constant__ CUtensorMap tmap_c, const Params p)
{
    static_assert(kRowB == ROW_BYTES || !Traits<kKind>::kBNMajor, "the finer ring is for K-major operands");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    PairCtrl *ctrl = reinterpret_cast<PairCtrl *>(smem + PAIR_STAGES * PAIR_STAGE_BYTES + EPI_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank & 1u) == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PAIR_MAX_STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctrl->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(&ctrl->tmem_full[a]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctrl->tmem_empty[a]), 8 * kWide);  // epilogue warps x 2 CTAs
        }
        ptx::mbar_init(ptx::smem_addr(&ctrl->acc_ready), 8 * kWide);
        ptx::mbar_init(ptx::smem_addr(&ctrl->mma_done), 1);
        ptx::mbar_init(ptx::smem_addr(&ctrl->never), 1);
        ctrl->wait.abort = 0;
        ctrl->wait.limit_ns = p.wait_limit_ns;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
        if (p.b3d) ptx::prefetch_tmap(&tmap_b2);
    }
    if (p.tma_store && warp == 2 && lane == 0) ptx::prefetch_tmap(&tmap_c);
    if (warp == PAIR_MMA_WARP) {
        ptx::tmem_alloc_pair(ptx::smem_addr(&ctrl->tmem_base), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // every CTA's barriers exist before any cross-CTA signal
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl->tmem_base;
    WaitCtl *wc = &ctrl->wait;
    const uint32_t smem_base = ptx::smem_addr(smem);

    if (warp == 0) {
        if (lane == 0) pair_producer<kKind, kWide, kRowB>(&tmap_a, &tmap_b, &tmap_b2, p, smem_base, ctrl, rank, wc);
    } else if (warp == PAIR_MMA_WARP) {
        if (leader) pair_mma<kKind, kWide, kRowB>(p, smem_base, ctrl, tmem_base, rank, lane, wc);
    } else if (warp == PAIR_WAITER_WARP) {
        if (leader) pair_waiter<kKind, kWide, kRowB>(p, ctrl, lane, wc);
    } else {
        pair_epilogue<kKind, kWide>(p, &tmap_c, ctrl, tmem_base, smem_base + PAIR_STAGES * PAIR_STAGE_BYTES,
                                     rank, warp, lane, wc);
    }

    __syncwarp();  // the barrier below is warp-aligned: reconverge lane 0 with the rest
    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while another may still signal or write it
    if (warp == PAIR_MMA_WARP) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------- CTA pairs for small M
//
// Problems of few rows (skinny M, a long K) are bound by the bytes every
// CTA pulls into shared memory: each CTA of the single-CTA kernel reloads
// all 128 rows of A for its 128 x bn tile.  Here a CTA pair shares one
// tcgen05.mma of M = 128 (cta_group::2): each CTA loads 64 rows of A and
// bn / 2 rows (or columns, N-major) of B per K block, so a tile of 128 x bn
// costs each CTA (64 + bn / 2) rows per K block instead of 128 + bn.  The
// accumulator of M = 128 lies in each CTA's TMEM as its 64 rows twice over:
// lanes 0-63 hold columns [0, bn / 2) and lanes 64-127 columns [bn / 2, bn),
// both in TMEM columns 0 .. bn / 2 - 1 (measured on GB300).
//   both CTAs  warp 0: TMA producer into the CTA's ring, two K blocks per
//              stage; both CTAs' loads complete on the leader's "full"
//              barrier, armed by the leader with the bytes of both;
//              warps 2-5: epilogue, warp w drains TMEM lane quarter w mod 4:
//              rows 32 (q mod 2) .. of the CTA's 64, column half q / 2;
//   leader     warp 1: the MMA issuer (one lane), committing each stage's
//              release to both CTAs' "empty" barriers and the finished
//              accumulator to both CTAs' "tmem_full".
// One tile per pair (a grid of 2 x tiles CTAs, at most one wave of pairs).
// p.bn is the tile width: 128, 192 or 256 (a multiple of 64 whose half is a
// whole number of B boxes); p.tiles_m counts 128-row bands.

constexpr int P128_A_BYTES = 64 * ROW_BYTES;  // 8 KB: this CTA's 64 rows of A, one K block
constexpr int P128_TMEM_COLS = 128;           // bn / 2 <= 128 accumulator columns

template <int kKind>
constexpr uint32_t p128_idesc(int bn)
{
    return (Traits<kKind>::kIdesc & ~(0x3Fu << 17) & ~(0x1Fu << 24)) |
           (static_cast<uint32_t>(bn >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

// Bytes one CTA loads for one K block (A rows, then B rows or columns).
__host__ __device__ constexpr uint32_t p128_half_bytes(int bn)
{
    return static_cast<uint32_t>(P128_A_BYTES + (bn / 2) * ROW_BYTES);
}

template <int kKind>
__device__ __forceinline__ void p128_producer(const CUtensorMap *tmap_a, const CUtensorMap *tmap_b,
                                              const CUtensorMap *tmap_b2, const Params &p, uint32_t smem_base,
                                              Ctrl *ctrl, uint32_t rank, WaitCtl *wc)
{
    using T = Traits<kKind>;
    const int64_t t = blockIdx.x / 2;
    const int64_t m0 = (t % p.tiles_m) * BM, n0 = (t / p.tiles_m) * p.bn;
    const int64_t mh = m0 + rank * 64, nb = n0 + rank * (p.bn / 2);  // this CTA's rows of A, of B
    const uint32_t half = p128_half_bytes(p.bn);
    uint32_t stage = 0, phase = 0, issued = 0, issued_phase = 0;
    bool ok = true;
    for (int64_t kb = 0; kb < p.num_kb; kb += 2) {
        if (!wait_bounded_cluster(ptx::smem_addr(&ctrl->empty[stage]), phase ^ 1u, wc)) {
            ok = false;
            break;
        }
        const bool second = kb + 1 < p.num_kb;
        const uint32_t full_local = ptx::smem_addr(&ctrl->full[stage]);
        const uint32_t full = ptx::mapa(full_local, 0);  // the leader's barrier
        if (rank == 0) ptx::mbar_arrive_expect_tx(full_local, (second ? 4u : 2u) * half);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1 && !second) break;
            const uint32_t sa = smem_base + stage * static_cast<uint32_t>(p.stage_bytes) + h * half;
            const uint32_t sb = sa + P128_A_BYTES;
            const int32_t kc = static_cast<int32_t>((kb + h) * T::BK);
            ptx::tma_load_2d_pair(sa, tmap_a, full, kc, static_cast<int32_t>(mh));
            if constexpr (!T::kBNMajor) {
                ptx::tma_load_2d_pair(sb, tmap_b, full, kc, static_cast<int32_t>(nb));
            } else if (p.b3d && nb + p.bn / 2 <= p.b3d_cols) {
                ptx::tma_load_3d_pair(sb, tmap_b, full, 0, kc, static_cast<int32_t>(nb / T::kNBox));
            } else {
                const CUtensorMap *m2 = p.b3d ? tmap_b2 : tmap_b;
#pragma unroll 1
                for (int c = 0; c < p.bn / 2 / T::kNBox; ++c)
                    ptx::tma_load_2d_pair(sb + c * T::kNBoxBytes, m2, full,
                                          static_cast<int32_t>(nb + c * T::kNBox), kc);
            }
        }
        issued |= 1u << stage;
        issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (!ok && rank == 0) {
        // the leader's barriers count both CTAs' bytes: wait (bounded) for
        // the loads in flight before the pair leaves
        for (int s = 0; s < p.stages; ++s)
            if ((issued >> s) & 1u) drain_wait(ptx::smem_addr(&ctrl->full[s]), (issued_phase >> s) & 1u);
    }
}

template <int kKind>
__device__ __forceinline__ void p128_mma(const Params &p, uint32_t smem_base, Ctrl *ctrl, uint32_t tmem_base,
                                         WaitCtl *wc)
{
    using T = Traits<kKind>;
    constexpr uint16_t kBoth = 0x3;
    const uint32_t half = p128_half_bytes(p.bn);
    const uint32_t idesc = p128_idesc<kKind>(p.bn);
    uint32_t stage = 0, phase = 0;
    bool ok = !p.inject_stall || wait_bounded(ptx::smem_addr(&ctrl->never), 0, wc);
    for (int64_t kb = 0; ok && kb < p.num_kb; kb += 2) {
        if (!wait_bounded_cluster(ptx::smem_addr(&ctrl->full[stage]), phase, wc)) {
            ok = false;
            break;
        }
        ptx::tc_fence_after();
        const bool second = kb + 1 < p.num_kb;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1 && !second) break;
            const uint32_t sa = smem_base + stage * static_cast<uint32_t>(p.stage_bytes) + h * half;
            const uint32_t sb = sa + P128_A_BYTES;
#pragma unroll
            for (int k = 0; k < T::BK / T::UMMA_K; ++k) {
                const uint64_t da = ptx::smem_desc(sa + k * 32, 16, 1024, ptx::kSw128);
                uint64_t db;
                if constexpr (!T::kBNMajor)
                    db = ptx::smem_desc(sb + k * 32, 16, 1024, ptx::kSw128);
                else
                    db = ptx::smem_desc(sb + k * T::kNStep, T::kNBoxBytes, T::kNSbo, T::kNLayout);
                ptx::umma_pair<kKind>(tmem_base, da, db, idesc, (kb + h != 0 || k != 0) ? 1u : 0u);
            }
        }
        ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->empty[stage]), kBoth);
        if (++stage == static_cast<uint32_t>(p.stages)) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (ok) ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->tmem_full[0]), kBoth);
    // every MMA this thread issued has finished before TMEM can be released
    ptx::umma_commit_pair_multicast(ptx::smem_addr(&ctrl->mma_done), 0x1);
    drain_wait(ptx::smem_addr(&ctrl->mma_done), 0);
}

template <int kKind>
__device__ __forceinline__ void p128_epilogue(const Params &p, const CUtensorMap *tmap_c, Ctrl *ctrl,
                                              uint32_t tmem_base, uint32_t epi_smem, uint32_t rank, int warp,
                                              int lane, WaitCtl *wc)
{
    const int64_t t = blockIdx.x / 2;
    const int64_t m0 = (t % p.tiles_m) * BM, n0 = (t / p.tiles_m) * p.bn;
    const uint32_t q = static_cast<uint32_t>(warp & 3);  // the TMEM lane quarter this warp may read
    const int cols = p.bn / 2;
    const int64_t row0 = m0 + rank * 64 + (q & 1u) * 32, col0 = n0 + (q >> 1) * cols;
    bool ok = wait_bounded_cluster(ptx::smem_addr(&ctrl->tmem_full[0]), 0, wc);
    ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
    if (ok) {
        ptx::tc_fence_after();
        uint32_t nbox = 0;
        // the tile lies inside C and the columns inside the allocation (warp-uniform)
        if (DGEMM_CHECK(m0 >= 0 && m0 < p.M && n0 >= 0 && n0 < p.N && cols <= P128_TMEM_COLS))
            drain_rows<kKind>(p, tmap_c, tmem_base + ((q * 32u) << 16), row0, col0,
                              epi_smem + q * 2 * EPI_BOX_BYTES, lane, nbox, cols);
    }
    if (lane == 0) ptx::bulk_wait<0>();  // stores done before the CTA leaves
}

template <int kKind>
__global__ void __launch_bounds__(cta_threads<true>(), 1)
    umma_pair128_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_b2, const __grid_constant__ CUtensorMap tmap_c,
                        const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + STAGES * STAGE_BYTES + EPI_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank() & 1u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < MAX_STAGES; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctrl->full[s]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctrl->empty[s]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&ctrl->tmem_full[0]), 1);
        ptx::mbar_init(ptx::smem_addr(&ctrl->mma_done), 1);
        ptx::mbar_init(ptx::smem_addr(&ctrl->never), 1);
        ctrl->wait.abort = 0;
        ctrl->wait.limit_ns = p.wait_limit_ns;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmap_a);
        ptx::prefetch_tmap(&tmap_b);
        if (p.b3d) ptx::prefetch_tmap(&tmap_b2);
    }
    if (p.tma_store && warp == 2 && lane == 0) ptx::prefetch_tmap(&tmap_c);
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(&ctrl->tmem_base), P128_TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctrl->tmem_base;
    WaitCtl *wc = &ctrl->wait;
    const uint32_t smem_base = ptx::smem_addr(smem);

    if (warp == 0) {
        if (lane == 0) p128_producer<kKind>(&tmap_a, &tmap_b, &tmap_b2, p, smem_base, ctrl, rank, wc);
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) p128_mma<kKind>(p, smem_base, ctrl, tmem_base, wc);
    } else {
        p128_epilogue<kKind>(p, &tmap_c, ctrl, tmem_base, smem_base + STAGES * STAGE_BYTES, rank, warp, lane,
                             wc);
    }

    __syncwarp();
    ptx::tc_fence_before();
    ptx::cluster_sync();  // no CTA leaves while the other may still signal or write it
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, P128_TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2-D tiled tensor map with a 128-byte swizzle and zero fill out of range.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D tiled map (dims innermost first; byte strides of dims 1 and 2), 128-
// byte swizzle family, zero fill out of range.
bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, const uint64_t (&dims)[3],
                 const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides[0], strides[1]};
    cuuint32_t b[3] = {box[0], box[1], box[2]};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kKind, bool kTma>
bool launch(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc, const Params &p,
            cudaStream_t stream, const DeviceInfo &dev)
{
    // the TMA kernel with two K blocks per stage is its own instance
    auto kernel = umma_gemm_kernel<kKind, kTma, 1>;
    if constexpr (kTma)
        if (p.kpb == 2) kernel = umma_gemm_kernel<kKind, true, 2>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
        return false;
    const int64_t tiles = p.tiles_m * p.tiles_n;
    const int64_t grid = tiles < dev.sm_count ? tiles : dev.sm_count;
    kernel<<<static_cast<unsigned>(grid), cta_threads<kTma>(), SMEM_BYTES, stream>>>(ma, mb, mc, p);
    return true;
}

// Co-resident clusters of the pair kernel (clusters of 2 CTAs) on the
// current device (0 if the kernel cannot run), cached per device and kind.
template <int kKind, int kWide = 1, int kRowB = ROW_BYTES>
int pair_clusters()
{
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices];
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::call_once(once[dev], [dev] {
        int n = 0;
        if (cudaFuncSetAttribute(umma_pair_kernel<kKind, kWide, kRowB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PAIR_SMEM_BYTES) == cudaSuccess) {
            int sms = 0;
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(sms - sms % 2));
            cfg.blockDim = dim3(pair_threads<kWide>());
            cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, umma_pair_kernel<kKind, kWide, kRowB>, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();  // a failed query leaves no sticky error behind
        cached[dev] = n;
    });
    return cached[dev];
}

// ---- stream-K workspace
//
// Static device memory of the library (no call allocates): a slot of partial
// sums per CTA pair (2 halves x 8 warp regions x 32 KB = 512 KB) for up to
// SK_MAX_PAIRS pairs, 64 MiB, and one 64-bit flag per region, zero from
// module load.  Launches that use it are ordered one after another, on
// whatever streams they come from, through an event that each records and
// the next waits for; each launch stamps its flags with a new generation, so
// flags left by earlier launches (or by an aborted one) never match.
// Stream-K is not used while the stream is being captured into a graph (the
// graph would hold the shared workspace); the round-robin schedule then
// runs, with bit-identical results.
__device__ __align__(256) float g_sk_work[SK_REGIONS * SK_REGION_FLOATS];
__device__ uint64_t g_sk_flags[SK_REGIONS];

struct SkWorkspace {
    std::mutex mu;
    float *work = nullptr;
    uint64_t *flags = nullptr;
    cudaEvent_t last = nullptr;
    bool recorded = false;
    bool failed = false;
    uint64_t gen = 0;
};

SkWorkspace *sk_workspace(int dev)
{
    constexpr int kMaxDevices = 64;
    static SkWorkspace ws[kMaxDevices];
    return dev >= 0 && dev < kMaxDevices ? &ws[dev] : nullptr;
}

// Resolve the current device's workspace for `slots` pairs (mu held).
bool sk_ensure(SkWorkspace &w, int64_t slots)
{
    if (slots > SK_MAX_PAIRS) return false;
    if (w.work) return true;
    if (w.failed) return false;
    void *work = nullptr, *flags = nullptr;
    cudaEvent_t ev = nullptr;
    if (cudaGetSymbolAddress(&work, g_sk_work) != cudaSuccess ||
        cudaGetSymbolAddress(&flags, g_sk_flags) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        w.failed = true;
        return false;
    }
    w.work = static_cast<float *>(work);
    w.flags = static_cast<uint64_t *>(flags);
    w.last = ev;
    return true;
}

bool stream_capturing(cudaStream_t stream)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
        cudaGetLastError();
        return true;  // cannot tell: take the schedule that needs no workspace
    }
    return st != cudaStreamCaptureStatusNone;
}

// Stream-K modes of the pair kernels (the `split` field of their tuning).
enum { kSkAuto = 0, kSkOff = 1, kSkOn = 2 };
// Estimated K-block time of one pair tile, 256 x 256 (us; x2 for 256 x 512):
// ~8.4 MFLOP (FP16, BK = 64) or ~4.2 MFLOP (TF32, BK = 32) at a pair's share
// of the measured rates (0.32 us for both on GB300).
constexpr double kSkKbUs = 0.32;
// Least estimated saving for a stream-K launch: the partials' round trip
// (a 256 KB store per CTA, and a load that the continuing pair's MMAs wait
// for) costs a few microseconds.
constexpr double kSkMinSavedUs = 8.0;

// Tiles of the stream-K region for T tiles on P pairs (0: whole tiles
// round-robin): P + T mod P when the tiles outnumber the pairs and the idle
// share of the last round is worth more than the partials cost.
int64_t stream_k_tiles(int64_t tiles, int64_t pairs, int64_t num_kb, double kb_us, int mode)
{
    if (mode == kSkOff || pairs < 2 || tiles <= pairs) return 0;
    const int64_t r = tiles % pairs;
    if (mode == kSkOn) return pairs + r;
    if (r == 0) return 0;
    const double saved_us = (1.0 - static_cast<double>(r) / static_cast<double>(pairs)) *
                            static_cast<double>(num_kb) * kb_us;
    return saved_us > kSkMinSavedUs ? pairs + r : 0;
}

// p.tiles_m / p.tiles_n count 256-row bands and tile columns (p.bn columns
// each).  sk_mode: kSkAuto / kSkOff / kSkOn.
// *sk tells whether the launch used stream-K.
template <int kKind, int kWide = 1, int kRowB = ROW_BYTES>
bool launch_pair(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mb2, const CUtensorMap &mc,
                 Params p, cudaStream_t stream, int sk_mode = kSkOff, bool *sk = nullptr)
{
    if (sk) *sk = false;
    const int clusters = pair_clusters<kKind, kWide, kRowB>();
    if (clusters <= 0) return false;
    const int64_t tiles = p.tiles_m * p.tiles_n;
    const int64_t n = tiles < clusters ? tiles : clusters;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * n));
    cfg.blockDim = dim3(pair_threads<kWide>());
    cfg.dynamicSmemBytes = PAIR_SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // (a K block of the finer ring is half as deep: half the time)
    p.sk_tiles = stream_k_tiles(tiles, n, p.num_kb, kSkKbUs * kWide * kRowB / ROW_BYTES, sk_mode);
    int dev = -1;
    SkWorkspace *w = nullptr;
    if (p.sk_tiles > 0 && !stream_capturing(stream) && cudaGetDevice(&dev) == cudaSuccess)
        w = sk_workspace(dev);
    if (w) {
        std::lock_guard<std::mutex> lock(w->mu);
        if (sk_ensure(*w, n)) {
            if (w->recorded && cudaStreamWaitEvent(stream, w->last, 0) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            p.sk_work = w->work;
            p.sk_flags = w->flags;
            p.sk_gen = ++w->gen;
            if (cudaLaunchKernelEx(&cfg, umma_pair_kernel<kKind, kWide, kRowB>, ma, mb, mb2, mc, p) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            w->recorded = cudaEventRecord(w->last, stream) == cudaSuccess;
            if (!w->recorded) cudaGetLastError();
            if (sk) *sk = true;
            return true;
        }
    }
    p.sk_tiles = 0;
    if (cudaLaunchKernelEx(&cfg, umma_pair_kernel<kKind, kWide, kRowB>, ma, mb, mb2, mc, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

template <int kKind>
int cluster_capacity(int size);

// The small-M pair kernel: one 128 x p.bn tile per pair, so at most one wave
// of co-resident pairs (false, nothing launched, beyond that).
template <int kKind>
bool launch_pair128(const CUtensorMap &ma64, const CUtensorMap &mb, const CUtensorMap &mb2, const CUtensorMap &mc,
                    const Params &p, cudaStream_t stream)
{
    const int64_t tiles = p.tiles_m * p.tiles_n;
    if (tiles < 1 || tiles > cluster_capacity<kKind>(2)) return false;
    if (cudaFuncSetAttribute(umma_pair128_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * tiles));
    cfg.blockDim = dim3(cta_threads<true>());
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, umma_pair128_kernel<kKind>, ma64, mb, mb2, mc, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// One-shot test hook (dgemm_test_inject_stall): applies to the next
// tensor-core launch made by this host thread.
thread_local uint64_t t_inject_limit_ns = 0;

Params make_params(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                   const void *B, int64_t ldb, float beta, void *C, int64_t ldc, int bk, bool vec_c)
{
    Params p;
    p.bn = BN;
    p.tma_store = 0;
    p.b3d = 0;
    p.b3d_cols = 0;
    p.sk_tiles = 0;
    p.sk_work = nullptr;
    p.sk_flags = nullptr;
    p.sk_gen = 0;
    p.stages = STAGES;
    p.stage_bytes = STAGE_BYTES;
    p.kpb = 1;
    const uint64_t stall = take_injected_stall();
    p.inject_stall = stall ? 1 : 0;
    p.splitk = 1;
    p.wait_limit_ns = stall ? stall : kWaitLimitNs;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.num_kb = (K + bk - 1) / bk;
    p.vec_c = vec_c ? 1 : 0;
    p.A = A;
    p.B = B;
    p.lda = lda;
    p.ldb = ldb;
    return p;
}

// Clusters of `size` CTAs of the single-CTA kernel that can be resident at
// once on the current device (0 if none), cached per device, kind and size.
template <int kKind>
int cluster_capacity(int size)
{
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices][9];
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    if (size < 2 || size > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    std::call_once(once[dev], [dev] {
        for (int s = 0; s < 9; ++s) cached[dev][s] = 0;
        if (cudaFuncSetAttribute(umma_gemm_kernel<kKind, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        for (int s = 2; s <= 8; ++s) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(s);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(sms - sms % s));
            cfg.blockDim = dim3(cta_threads<true>());
            cfg.dynamicSmemBytes = SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, umma_gemm_kernel<kKind, true>, &cfg) != cudaSuccess)
                n = 0;
            cached[dev][s] = n;
        }
        cudaGetLastError();
    });
    return cached[dev][size];
}

// Split factor for problems with few output tiles: the largest S <= 8 (the
// portable cluster size) such that every range has at least 8 K blocks and
// all tiles x S CTAs are resident in one wave of clusters.  1 = no split.
// Tile configuration of one call: the CTA-pair kernel (256 x 256 tiles), the
// persistent single-CTA kernel (128 x bn tiles) or split-K over S CTAs of a
// cluster (128 x bn tiles).
// (4 is unused: it once named a two-pair cluster variant, since removed.)
// 6 and 7: the pair kernels with the finer ring (32-deep K stages of the
// K-major 16-bit kinds, see PairShape).
// 8: the CTA pair for small M (128 x bn tiles, 64 rows of A per CTA).
enum { kVariantAuto = 0, kVariantPair = 1, kVariantSingle = 2, kVariantSplit = 3, kVariantWide = 5,
       kVariantPairFine = 6, kVariantWideFine = 7, kVariantPair128 = 8 };
struct UmmaConfig {
    int variant;
    int bn;
    int split;
};

// One-shot override of the next call on this host thread (dgemm_tune_next).
thread_local UmmaConfig t_tune = {kVariantAuto, BN, 1};

// Narrowest tile width step of a kind: the N-major 16-bit kinds load B in
// 64-column boxes; the others take any multiple of 32.
template <int kKind>
constexpr int bn_step()
{
    return Traits<kKind>::kBNMajor ? Traits<kKind>::kNBox : 32;
}

// Automatic choice.  Problems with more than half a wave of 128 x 256 tiles
// take the pair kernel (M > 128; else the single-CTA kernel, 256 wide).
// Smaller ones -- skinny M, or few tiles and a long K -- choose the
// tile width bn and the split S that keep the most SMs streaming:
//   * candidates: bn from 256 down in the kind's step (32, or 64 for the
//     16-bit NN kinds); S from 1 to 8 with at least 8 K blocks per rank,
//     tiles * S <= SMs, and all clusters resident at once;
//   * estimated time = its K blocks x max(MMA time, load time) per CTA +
//     the cost of adding S partials, with the load time of a K block
//     (128 + bn rows of 128 bytes) at a per-CTA stream rate, and the whole
//     launch no faster than the operands at the HBM rate nor than all the
//     CTAs' stage bytes at an aggregate L2 -> SM rate;
//   * the smallest estimate wins (ties: the wider tile, the smaller S).
// The constants are fitted to GB300 sweeps of the tuning tool
// (dense_gemm_09_gb300/tune.py, 15 shapes; every automatic choice within
// 2 % of the best configuration measured): an MMA K block of 128 x 256 x
// 128 bytes in ~0.33 us; a CTA streams ~65 GB/s with one K block per stage
// and ~100 GB/s with two (tiles up to 128 wide, see set_ring); HBM ~6 TB/s;
// L2 -> SM ~10 TB/s in all; a split costs ~1 us plus ~0.25 us per extra
// rank plus ~0.5 us per 64 KB of partials moved.
template <int kKind>
UmmaConfig choose_config(const Params &p, int sm_count, bool pair_ok)
{
    using T = Traits<kKind>;
    const int64_t tiles256 = p.tiles_m * ((p.N + BN - 1) / BN);
    // more than half a wave of 128 x 256 tiles: the pair halves each CTA's
    // operand traffic (2048^3: FP16 21.3 us pair, 22.0 us single; TF32 31.4
    // and 34.6 us)
    // Problems of more than half a wave of 128 x 256 tiles take a CTA-pair
    // kernel, with 256 x 256 or 256 x 512 tiles, each with whole tiles dealt
    // round-robin or with a stream-K tail.  Estimated time, with P pairs,
    // T tiles and t the time of a 256 x 256 tile (num_kb K blocks):
    //   round-robin  ceil(T / P) x t_tile
    //   stream-K     T / P x t_tile + the partials' cost
    // A 256 x 512 tile takes 2 x f x t: it carries a quarter fewer operand
    // bytes per flop into each SM, worth f = 0.97 for TF32; the power-bound
    // 16-bit kinds gain nothing per tile (f = 1).  Stream-K costs ~8 us with
    // 256 x 256 tiles and, with 256 x 512 tiles (one accumulator, so every
    // extra unit of work stalls the MMAs for a drain), ~3 + 5 x (bytes per C
    // element) us.  Fitted to GB300 sweeps (8192 x 8192 x 4096, n^3 for n =
    // 4096, 12288, 16384, 8192 x 8448 x 4096, FP16 and TF32); ties go to
    // the earlier of wide / pair round-robin, wide / pair stream-K.
    if (pair_ok && p.M > BM && tiles256 * 2 > sm_count) {
        const int64_t pairs = sm_count / 2;
        const int64_t bands = (p.M + PAIR_BM - 1) / PAIR_BM;
        const int64_t tp = bands * ((p.N + BN - 1) / BN), tw = bands * ((p.N + 2 * BN - 1) / (2 * BN));
        const double t = static_cast<double>(p.num_kb) * kSkKbUs;
        const double f = T::kElem == 4 ? 0.97 : 1.0;
        const double ovh_w = 3.0 + 5.0 * (T::kElem == 4 ? 4 : 2), ovh_p = 8.0;
        auto rr = [&](int64_t tiles) { return static_cast<double>((tiles + pairs - 1) / pairs); };
        auto fr = [&](int64_t tiles) { return static_cast<double>(tiles) / static_cast<double>(pairs); };
        const bool sk_w = tw > pairs && tw % pairs != 0, sk_p = tp > pairs && tp % pairs != 0;
        struct Cand {
            double us;
            UmmaConfig cfg;
        } cand[4] = {
            {rr(tw) * 2.0 * f * t, {kVariantWide, BN, kSkOff}},
            {rr(tp) * t, {kVariantPair, BN, kSkOff}},
            {sk_w ? fr(tw) * 2.0 * f * t + ovh_w : 1e30, {kVariantWide, BN, kSkOn}},
            {sk_p ? fr(tp) * t + ovh_p : 1e30, {kVariantPair, BN, kSkOn}},
        };
        int best = 0;
        for (int i = 1; i < 4; ++i)
            if (cand[i].us < cand[best].us * 0.995) best = i;
        return cand[best].cfg;
    }
    if (tiles256 * 2 > sm_count) return {kVariantSingle, BN, 1};
    const double kb_mma_us = 0.33 / 256.0;          // per column of bn, one K block
    const double cta_bytes_per_us_1 = 65e3;         // 65 GB/s, one K block per stage
    const double cta_bytes_per_us_2 = 100e3;        // 100 GB/s, two (bn <= 128)
    const double hbm_bytes_per_us = 6.0e6;          // 6 TB/s
    const double l2_bytes_per_us = 10.0e6;          // 10 TB/s, L2 -> all SMs
    const double operand_bytes = static_cast<double>(p.M * p.K + p.N * p.K) * T::kElem;
    UmmaConfig best{kVariantSingle, BN, 1};
    double best_t = 1e30;
    for (int bn = BN; bn >= bn_step<kKind>(); bn -= bn_step<kKind>()) {
        const int64_t tiles = p.tiles_m * ((p.N + bn - 1) / bn);
        const double rate = bn * ROW_BYTES <= 16 * 1024 ? cta_bytes_per_us_2 : cta_bytes_per_us_1;
        for (int S = 1; S <= 8; ++S) {
            if (tiles * S > sm_count) break;
            if (S > 1 && (p.num_kb < 8 * S || tiles > cluster_capacity<kKind>(S))) continue;
            const int64_t kb = (p.num_kb + S - 1) / S;
            const double kb_bytes = (BM + bn) * 128.0;
            const double t_kb = std::max(kb_mma_us * bn, kb_bytes / rate);
            double t = std::max({kb * t_kb, operand_bytes / hbm_bytes_per_us,
                                 static_cast<double>(tiles * S * kb) * kb_bytes / l2_bytes_per_us});
            if (S > 1) t += 1.0 + 0.25 * (S - 1) + 0.5 * (BM * bn * 4.0 / 65536.0) * (S - 1) / S;
            if (t < best_t * 0.98) {
                best_t = t;
                best = {S > 1 ? kVariantSplit : kVariantSingle, bn, S};
            }
        }
    }
    // The small-M pair, by rule rather than by the model (its per-CTA stream
    // rate is lower than the single-CTA kernel's: both CTAs' loads, and a
    // round trip between them, gate every stage): 16-bit kinds, one band of
    // rows and 48 to 76 tiles of 128 x 256, where it measured faster than
    // every configuration above (FP16 127 x 12288 x 4096: TN 26.6 against
    // 26.9 us, NN 26.8 against 28.6 us; TF32 and fewer tiles were slower).
    if constexpr (!T::kTf32) {
        const int64_t tiles = (p.N + BN - 1) / BN;
        if (p.tiles_m == 1 && tiles >= 48 && tiles * 2 <= sm_count && tiles <= cluster_capacity<kKind>(2))
            return {kVariantPair128, BN, 1};
    }
    return best;
}

template <int kKind>
bool launch_splitk(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                   const Params &p, cudaStream_t stream)
{
    auto kernel = p.kpb == 2 ? umma_gemm_kernel<kKind, true, 2> : umma_gemm_kernel<kKind, true, 1>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.splitk);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.tiles_m * p.tiles_n * p.splitk));
    cfg.blockDim = dim3(cta_threads<true>());
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, ma, mb, mc, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// Variant names ("umma_<kind>_<variant>"), built once per kind:
// [0] pair, [1] register / cp.async producer, then per tile width bn
// (32..256) the single-CTA TMA kernel and split-K S = 2..8.
template <int kKind>
const char *variant_name(int variant, int bn = BN, int split = 1, bool sk = false)
{
    static std::string names[10 + 9 * 9 + 9];  // [2 + 9 * 9] and [10 + 9 * 9] unused
    static std::once_flag once;
    std::call_once(once, [] {
        using T = Traits<kKind>;
        const char *kind = kKind == kF16 ? "f16_tn" : kKind == kTF32 ? "tf32" : kKind == kBF16 ? "bf16_tn"
                         : kKind == kF16NN ? "f16_nn" : "bf16_nn";
        const std::string bk = std::to_string(T::BK);
        const std::string base = std::string("umma_") + kind;
        names[0] = base + "_pair_256x256x" + bk + "_tma";
        names[3 + 9 * 9] = base + "_pair_256x512x" + bk + "_tma";
        names[4 + 9 * 9] = base + "_pair_256x256x" + bk + "_sk_tma";
        names[5 + 9 * 9] = base + "_pair_256x512x" + bk + "_sk_tma";
        const std::string bkf = std::to_string(64 / T::kElem);  // the finer ring's K per stage
        names[6 + 9 * 9] = base + "_pair_256x256x" + bkf + "_tma";
        names[7 + 9 * 9] = base + "_pair_256x256x" + bkf + "_sk_tma";
        names[8 + 9 * 9] = base + "_pair_256x512x" + bkf + "_tma";
        names[9 + 9 * 9] = base + "_pair_256x512x" + bkf + "_sk_tma";
        names[1] = base + "_128x256x" + bk + (kKind == kTF32 ? "_cpasync" : "_ldst");
        for (int w = 1; w <= 8; ++w) {
            const std::string tile = "128x" + std::to_string(32 * w) + "x" + bk;
            names[2 + w * 9 + 1] = base + "_" + tile + "_tma";
            for (int S = 2; S <= 8; ++S)
                names[2 + w * 9 + S] = base + "_splitk" + std::to_string(S) + "_" + tile + "_tma";
            names[10 + 9 * 9 + w] = base + "_pair_" + tile + "_tma";
        }
    });
    if (variant == kVariantPair128) return names[10 + 9 * 9 + bn / 32].c_str();
    if (variant == kVariantPair) return names[sk ? 4 + 9 * 9 : 0].c_str();
    if (variant == kVariantWide) return names[sk ? 5 + 9 * 9 : 3 + 9 * 9].c_str();
    if (variant == kVariantPairFine) return names[sk ? 7 + 9 * 9 : 6 + 9 * 9].c_str();
    if (variant == kVariantWideFine) return names[sk ? 9 + 9 * 9 : 8 + 9 * 9].c_str();
    if (variant == kVariantAuto) return names[1].c_str();  // the non-TMA kernel
    const int w = bn / 32, S = variant == kVariantSplit ? split : 1;
    return names[2 + w * 9 + S].c_str();
}

// The single-CTA TMA kernel's ring for tile width p.bn: as many stages as
// fit in the ring space (at most MAX_STAGES), each of kpb K blocks of
// A_TILE_BYTES + bn * ROW_BYTES.  Two K blocks per stage for tiles up to
// 128 wide (a block's B at most 16 KB).  Measured on GB300, a plain TMA
// stream whose stages carry 16 KB runs ~20 % slower than one whose stages
// carry 32 KB, however many stages are in flight: a fixed cost per stage,
// which the deeper stages halve (with the kernel's code cached: 256^3 FP16
// 10.2 -> 8.6 us, 1024^3 14.3 -> 12.3 us, 512 x 512 x 8192 22.5 -> 20.6 us,
// TF32 64 x 2048 x 8192 28.6 -> 25.9 us; at 160 wide, three stages of two
// blocks were slower than five of one).  Split-K launches do not use the
// epilogue boxes (their partials meet in the ring), so their ring may extend
// over them.
void set_ring(Params &p, bool split)
{
    const int half = A_TILE_BYTES + p.bn * ROW_BYTES;
    const int space = STAGES * STAGE_BYTES + (split ? EPI_BYTES : 0);
    p.kpb = p.bn * ROW_BYTES <= 16 * 1024 ? 2 : 1;
    p.stage_bytes = p.kpb * half;
    p.stages = std::min(MAX_STAGES, space / p.stage_bytes);
}

// TMA-capable operands.  ma: A with 128-row boxes; mb_pair: B boxes of the
// pair kernel (null if B cannot be described); make_b(bn, map) builds B's map
// for 128 x bn tiles; make_a64(map) A's map with 64-row boxes.
template <int kKind, typename MakeB, typename MakeA64>
const char *dispatch_tma(const Params &p0, const CUtensorMap &ma, const CUtensorMap *mb_pair,
                         const CUtensorMap *mb_pair2, const CUtensorMap *ma_fine, const CUtensorMap *mb_fine,
                         int pair3d, int64_t pair3d_cols, MakeB make_b, MakeA64 make_a64, const CUtensorMap &mc,
                         cudaStream_t stream, const DeviceInfo &dev)
{
    UmmaConfig cfg = t_tune;
    t_tune = UmmaConfig{kVariantAuto, BN, 1};
    // the finer ring needs its own tensor maps (K-major 16-bit operands);
    // without them a request for it takes the ordinary ring
    if (cfg.variant == kVariantPairFine && !(ma_fine && mb_fine)) cfg.variant = kVariantPair;
    if (cfg.variant == kVariantWideFine && !(ma_fine && mb_fine)) cfg.variant = kVariantWide;
    if (((cfg.variant == kVariantPair || cfg.variant == kVariantWide) && !mb_pair) || cfg.bn % bn_step<kKind>() != 0)
        cfg.variant = kVariantAuto;
    // every rank of a split needs at least one K block
    if (cfg.variant == kVariantSplit && cfg.split > p0.num_kb)
        cfg = p0.num_kb >= 2 ? UmmaConfig{kVariantSplit, cfg.bn, static_cast<int>(p0.num_kb)}
                             : UmmaConfig{kVariantSingle, cfg.bn, 1};
    if (cfg.variant == kVariantAuto)
        cfg = choose_config<kKind>(p0, dev.sm_count, mb_pair != nullptr);
    if (cfg.variant == kVariantPair128) {
        // the small-M pair: B in boxes of bn / 2 rows (columns, N-major)
        Params q = p0;
        q.bn = cfg.bn;
        q.tiles_m = (p0.M + BM - 1) / BM;
        q.tiles_n = (p0.N + cfg.bn - 1) / cfg.bn;
        q.stage_bytes = 2 * static_cast<int>(p128_half_bytes(cfg.bn));
        q.stages = std::min(MAX_STAGES, STAGES * STAGE_BYTES / q.stage_bytes);
        if ((cfg.bn / 2) % box_cols<kKind>() != 0) q.tma_store = 0;
        CUtensorMap a64{}, bh{};
        int b3d = 0;
        const bool fits = !Traits<kKind>::kBNMajor || (cfg.bn / 2) % Traits<kKind>::kNBox == 0;
        if (fits && make_a64(&a64) && make_b(cfg.bn / 2, &bh, &b3d)) {
            q.b3d = b3d;
            q.b3d_cols = b3d ? INT64_MAX : 0;
            if (launch_pair128<kKind>(a64, bh, bh, mc, q, stream)) return variant_name<kKind>(kVariantPair128, cfg.bn);
        }
        // (a tile count beyond one wave of pairs, or a B the boxes cannot
        // describe): the automatic choice among the other kernels
        cfg = choose_config<kKind>(p0, dev.sm_count, mb_pair != nullptr);
        if (cfg.variant == kVariantPair128) cfg = UmmaConfig{kVariantSingle, BN, 1};
    }
    Params p = p0;
    if constexpr (!Traits<kKind>::kBNMajor) {
        if (cfg.variant == kVariantPairFine || cfg.variant == kVariantWideFine) {
            const bool wide = cfg.variant == kVariantWideFine;
            Params f = p;
            f.tiles_m = (p.M + PAIR_BM - 1) / PAIR_BM;
            f.b3d = 0;
            f.num_kb = (p.K + 64 / Traits<kKind>::kElem - 1) / (64 / Traits<kKind>::kElem);  // 32-deep K blocks
            if (wide) {
                f.bn = 2 * BN;  // 256 x 512 pair tiles
                f.tiles_n = (p.N + 2 * BN - 1) / (2 * BN);
                if (f.bn % box_cols<kKind>() != 0) f.tma_store = 0;
            }
            bool sk = false;
            const bool ok = wide ? launch_pair<kKind, 2, 64>(*ma_fine, *mb_fine, *mb_fine, mc, f, stream, cfg.split, &sk)
                                 : launch_pair<kKind, 1, 64>(*ma_fine, *mb_fine, *mb_fine, mc, f, stream, cfg.split, &sk);
            if (ok) return variant_name<kKind>(cfg.variant, BN, 1, sk);
            cfg.variant = wide ? kVariantWide : kVariantPair;
        }
    }
    if (cfg.variant == kVariantPair || cfg.variant == kVariantWide) {
        p.tiles_m = (p.M + PAIR_BM - 1) / PAIR_BM;
        p.b3d = pair3d;
        p.b3d_cols = pair3d_cols;
        bool sk = false;
        if (cfg.variant == kVariantWide) {
            Params w = p;
            w.bn = 2 * BN;  // 256 x 512 pair tiles
            w.tiles_n = (p.N + 2 * BN - 1) / (2 * BN);
            if (w.bn % box_cols<kKind>() != 0) w.tma_store = 0;
            if (launch_pair<kKind, 2>(ma, *mb_pair, *mb_pair2, mc, w, stream, cfg.split, &sk))
                return variant_name<kKind>(kVariantWide, BN, 1, sk);
        }
        if (launch_pair<kKind, 1>(ma, *mb_pair, *mb_pair2, mc, p, stream, cfg.split, &sk))
            return variant_name<kKind>(kVariantPair, BN, 1, sk);
        cfg = UmmaConfig{kVariantSingle, BN, 1};
        p = p0;
    }
    p.bn = cfg.bn;
    p.tiles_n = (p.N + cfg.bn - 1) / cfg.bn;
    if (p.bn % box_cols<kKind>() != 0) p.tma_store = 0;
    CUtensorMap mb{};
    int b3d = 0;
    if (!make_b(cfg.bn, &mb, &b3d)) return nullptr;
    p.b3d = b3d;
    if (cfg.variant == kVariantSplit) {
        p.splitk = cfg.split;
        set_ring(p, true);
        if (launch_splitk<kKind>(ma, mb, mc, p, stream))
            return variant_name<kKind>(kVariantSplit, cfg.bn, cfg.split);
        p.splitk = 1;
    }
    set_ring(p, false);
    return launch<kKind, true>(ma, mb, mc, p, stream, dev) ? variant_name<kKind>(kVariantSingle, cfg.bn)
                                                           : nullptr;
}

template <int kKind>
constexpr bool T_is_n_major()
{
    return Traits<kKind>::kBNMajor;
}

template <int kKind>
const char *launch_kind(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                        const void *B, int64_t ldb, float beta, void *C, int64_t ldc,
                        cudaStream_t stream, const DeviceInfo &dev, int64_t n_b)
{
    // columns of an N-major B the loads may cover (zeros past N)
    const int64_t NB = T_is_n_major<kKind>() && n_b > N ? n_b : N;
    using T = Traits<kKind>;
    constexpr int es = T::kElem;
    const CUtensorMapDataType dt = T::kTf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : T::kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    Params p = make_params(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, T::BK,
                           aligned16(C) && (ldc * es) % 16 == 0);
    CUtensorMap mc{};
    p.tma_store = (p.vec_c && make_map(&mc, dt, C, N, M, ldc * es, box_cols<kKind>(), 32,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
                      ? 1 : 0;
    // TMA needs 16-byte aligned bases and row pitches.
    const bool tma = aligned16(A) && aligned16(B) && (lda * es) % 16 == 0 && (ldb * es) % 16 == 0;
    CUtensorMap ma{}, mbp{};
    if (tma && make_map(&ma, dt, A, K, M, lda * es, T::BK, BM, CU_TENSOR_MAP_SWIZZLE_128B)) {
        // B stored N x K: bn-row boxes (single CTA), 128-row boxes (pair).
        // B stored K x N (N-major): when N is a whole number of 128-byte
        // column groups, one 3-D box per stage -- B viewed as [N / kNBox
        // groups][K rows][kNBox columns], a box of bn / kNBox groups -- which
        // lands in the same shared-memory layout as bn / kNBox 2-D boxes of 128
        // bytes x BK rows, in one instruction; otherwise the 2-D boxes (a
        // partial last group would read past the end of B's rows).
        auto make_b = [&](int bn, CUtensorMap *m, int *b3d) {
            *b3d = 0;
            if constexpr (T::kBNMajor) {
                const CUtensorMapSwizzle sw =
                    T::kTf32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
                if (NB % T::kNBox == 0 &&
                    make_map_3d(m, dt, B,
                                {static_cast<uint64_t>(T::kNBox), static_cast<uint64_t>(K),
                                 static_cast<uint64_t>(NB / T::kNBox)},
                                {static_cast<uint64_t>(ldb * es), static_cast<uint64_t>(T::kNBox * es)},
                                {static_cast<uint32_t>(T::kNBox), static_cast<uint32_t>(T::BK),
                                 static_cast<uint32_t>(bn / T::kNBox)},
                                sw)) {
                    *b3d = 1;
                    return true;
                }
                return make_map(m, dt, B, NB, K, ldb * es, T::kNBox, T::BK, sw);
            } else {
                return make_map(m, dt, B, K, N, ldb * es, T::BK, bn, CU_TENSOR_MAP_SWIZZLE_128B);
            }
        };
        CUtensorMap probe{};
        int probe3d = 0, pair3d = 0;
        if (make_b(BN, &probe, &probe3d)) {
            bool ok_pair = make_b(128, &mbp, &pair3d);
            // a 3-D map over every column group serves every half (groups past
            // it read as zeros); mbp2 is then never used
            int64_t pair3d_cols = pair3d ? INT64_MAX : 0;
            CUtensorMap mbp2 = mbp;
            if constexpr (T::kBNMajor) {
                // N not a whole number of column groups: the pair kernels still
                // load every tile column but the last with one 3-D box per stage,
                // from a 3-D map over the whole groups; the last takes 2-D boxes
                // (mbp, the 2-D map over all of B)
                const int64_t whole = NB / T::kNBox * T::kNBox;
                const CUtensorMapSwizzle sw =
                    T::kTf32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
                CUtensorMap m3{};
                if (ok_pair && !pair3d && whole >= 128 &&
                    make_map_3d(&m3, dt, B,
                                {static_cast<uint64_t>(T::kNBox), static_cast<uint64_t>(K),
                                 static_cast<uint64_t>(whole / T::kNBox)},
                                {static_cast<uint64_t>(ldb * es), static_cast<uint64_t>(T::kNBox * es)},
                                {static_cast<uint32_t>(T::kNBox), static_cast<uint32_t>(T::BK),
                                 static_cast<uint32_t>(128 / T::kNBox)},
                                sw)) {
                    mbp2 = mbp;
                    mbp = m3;
                    pair3d = 1;
                    pair3d_cols = whole;
                }
            }
            // the finer ring (K-major 16-bit kinds, only on request through the
            // tuning hook): 32-element boxes under the 64-byte swizzle
            CUtensorMap maf{}, mbf{};
            bool ok_fine = false;
            if constexpr (!T::kBNMajor && T::kElem == 2)
                if (t_tune.variant == kVariantPairFine || t_tune.variant == kVariantWideFine)
                    ok_fine = make_map(&maf, dt, A, K, M, lda * es, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) &&
                              make_map(&mbf, dt, B, K, N, ldb * es, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B);
            auto make_a64 = [&](CUtensorMap *m) {
                return make_map(m, dt, A, K, M, lda * es, T::BK, 64, CU_TENSOR_MAP_SWIZZLE_128B);
            };
            return dispatch_tma<kKind>(p, ma, ok_pair ? &mbp : nullptr, ok_pair ? &mbp2 : nullptr,
                                       ok_fine ? &maf : nullptr, ok_fine ? &mbf : nullptr, pair3d, pair3d_cols,
                                       make_b, make_a64, mc, stream, dev);
        }
    }
    t_tune = UmmaConfig{kVariantAuto, BN, 1};
    CUtensorMap mb{};
    return launch<kKind, false>(ma, mb, mc, p, stream, dev) ? variant_name<kKind>(kVariantAuto) : nullptr;
}

}  // namespace

const char *launch_umma(int kind, int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                        int64_t lda, const void *B, int64_t ldb, float beta, void *C, int64_t ldc,
                        cudaStream_t stream, const DeviceInfo &dev, int64_t n_b)
{
    switch (kind) {
    case kUmmaF16TN:
        return launch_kind<kF16>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev, n_b);
    case kUmmaTF32NN:
        return launch_kind<kTF32>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev, n_b);
    case kUmmaBF16TN:
        return launch_kind<kBF16>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev, n_b);
    case kUmmaF16NN:
        return launch_kind<kF16NN>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev, n_b);
    case kUmmaBF16NN:
        return launch_kind<kBF16NN>(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, dev, n_b);
    default:
        return nullptr;
    }
}

int umma_tune_next(int variant, int bn, int split)
{
    if (variant < kVariantAuto || variant > kVariantPair128 || variant == 4) return DGEMM_ERR_INVALID_ARG;
    if (variant == kVariantPair128 && (bn < 128 || bn > BN || bn % 64 != 0)) return DGEMM_ERR_INVALID_ARG;
    if ((variant == kVariantSingle || variant == kVariantSplit) && (bn < 32 || bn > BN || bn % 32 != 0))
        return DGEMM_ERR_INVALID_ARG;
    if (variant == kVariantSplit && (split < 2 || split > 8)) return DGEMM_ERR_INVALID_ARG;
    const bool paired = variant == kVariantPair || variant == kVariantWide || variant == kVariantPairFine ||
                        variant == kVariantWideFine;
    if (paired && (split < kSkAuto || split > kSkOn)) return DGEMM_ERR_INVALID_ARG;
    const bool sized = variant == kVariantSingle || variant == kVariantSplit || variant == kVariantPair128;
    t_tune = UmmaConfig{variant, sized ? bn : BN, variant == kVariantSplit || paired ? split : 1};
    return DGEMM_OK;
}

// ---- test hooks: the host-compiled schedule and tile choice (no launch)

int64_t umma_test_pair_units(int64_t tiles, int64_t pairs, int64_t num_kb, int64_t sk_tiles, int64_t pair,
                             int64_t *out, int64_t max_units)
{
    if (tiles < 1 || pairs < 1 || num_kb < 1 || pair < 0 || pair >= pairs || sk_tiles < 0 || sk_tiles > tiles ||
        (sk_tiles > 0 && sk_tiles < pairs) || max_units < 0 || (max_units > 0 && !out))
        return -1;
    Params p{};
    p.tiles_m = tiles;  // a 1-D tile order is all the schedule sees
    p.tiles_n = 1;
    p.num_kb = num_kb;
    p.sk_tiles = sk_tiles;
    WorkIter it(p, pair, pairs);
    Unit u;
    int64_t n = 0;
    while (it.next(p, u)) {
        if (n < max_units) {
            int64_t *o = out + 5 * n;
            o[0] = u.t;
            o[1] = u.k0;
            o[2] = u.k1;
            o[3] = u.init ? 1 : 0;
            o[4] = u.publish ? 1 : 0;
        }
        ++n;
    }
    return n;
}

int64_t umma_test_stream_k_tiles(int64_t tiles, int64_t pairs, int64_t num_kb, int wide, int mode)
{
    if (wide < 1 || wide > 2 || mode < kSkAuto || mode > kSkOn) return -1;
    return stream_k_tiles(tiles, pairs, num_kb, kSkKbUs * wide, mode);
}

template <int kKind>
UmmaConfig test_choose(int64_t M, int64_t N, int64_t K, int sm_count)
{
    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.bn = BN;
    p.tiles_m = (M + BM - 1) / BM;
    p.tiles_n = (N + BN - 1) / BN;
    p.num_kb = (K + Traits<kKind>::BK - 1) / Traits<kKind>::BK;
    return choose_config<kKind>(p, sm_count, true);
}

int umma_test_choose(int kind, int64_t M, int64_t N, int64_t K, int sm_count, int *variant, int *bn, int *split)
{
    if (M < 1 || N < 1 || K < 1 || sm_count < 2 || !variant || !bn || !split) return DGEMM_ERR_INVALID_ARG;
    UmmaConfig c;
    switch (kind) {
    case kF16: c = test_choose<kF16>(M, N, K, sm_count); break;
    case kTF32: c = test_choose<kTF32>(M, N, K, sm_count); break;
    case kBF16: c = test_choose<kBF16>(M, N, K, sm_count); break;
    case kF16NN: c = test_choose<kF16NN>(M, N, K, sm_count); break;
    case kBF16NN: c = test_choose<kBF16NN>(M, N, K, sm_count); break;
    default: return DGEMM_ERR_INVALID_ARG;
    }
    cudaGetLastError();  // the capacity queries of small problems fail without a GPU
    *variant = c.variant;
    *bn = c.bn;
    *split = c.split;
    return DGEMM_OK;
}

void umma_inject_stall(uint64_t wait_limit_ns)
{
    t_inject_limit_ns = wait_limit_ns ? wait_limit_ns : 1;
}

uint64_t take_injected_stall()
{
    const uint64_t v = t_inject_limit_ns;
    t_inject_limit_ns = 0;
    return v;
}

bool encode_tiled_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle)
{
    return make_map(m, dt, base, inner, outer, row_bytes, box_inner, box_outer, swizzle);
}

int umma_read_status(int clear)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_umma_status, sizeof(int)) != cudaSuccess) return DGEMM_ERR_LAUNCH;
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_umma_status, &zero, sizeof(int)) != cudaSuccess)
            return DGEMM_ERR_LAUNCH;
    }
    return v;
}

}  // namespace dgemm

DGEMM_DEFINE_CHECK_READER(check_status_umma)
