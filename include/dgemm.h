/*
 * dgemm.h -- C ABI of libdgemm, a dense row-major GEMM library for one
 * NVIDIA GB300 (compute capability 10.3, sm_103a).
 *
 * Every entry point computes
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * on the GPU, asynchronously on the caller's CUDA stream, and returns a
 * dgemm_status.  The operation is the one the pages define:
 *   - "CUDA GEMM：从基础写法到工程优化", opening definition: C = alpha*A*B +
 *     beta*C with A (M x K), B (K x N), C (M x N), all row-major;
 *   - "SGEMM CUDA代码学习", section "问题定义与记号": A[m][k] sits at m*K + k,
 *     and one output element is one K-long dot product;
 *   - "Warp Specialization HGEMM", section "6. B 的 RowMajor(K,N) 与 TN 布局":
 *     the TN layout, where B is stored N x K (row-major) and the product is
 *     A * B^T.
 * The pages' matrices are tight (leading dimension = row length); this ABI
 * adds explicit leading dimensions (lda, ldb, ldc, in elements).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: the caller owns every buffer.  A and B are device pointers that
 *   are only read (never modified, not even to round them).  C is a device
 *   pointer; it is read only when beta != 0 and it is always written (all
 *   M x N entries, nothing outside them -- padding columns between N and ldc
 *   are left untouched).
 * Memory: no call allocates device memory or synchronises; results are
 *   ready when the stream reaches the call.  The library keeps a per-device
 *   cache of device properties, and two arrays of static device memory
 *   (allocated with the library's code when it is loaded): the 64 MiB
 *   scratch of gemm_tf32_noalloc and the 64 MiB stream-K workspace of the
 *   tensor-core calls.
 * Stream-K: when a large problem's output tiles do not divide evenly over
 *   the CTA pairs, the tensor-core calls may cut the first tiles along K
 *   (one contiguous range of K blocks per pair).  The pair that finishes a
 *   cut tile starts from the raw FP32 partial sum the previous pair left in
 *   the workspace, so results are bit-identical to uncut tiles.  Launches
 *   that use the workspace are ordered one after another across streams
 *   through an event (the library records it and makes the next such launch
 *   wait on it); under stream capture the calls do not cut tiles.  So two
 *   tensor-core calls on different, otherwise independent streams do not
 *   overlap on the GPU when both cut tiles: the one issued second starts
 *   after the first has finished (each result is still exact).  Calls that
 *   do not cut tiles, and gemm_f32, are not ordered this way.  Source: none
 *   on the pages (their kernels deal whole tiles).
 * Special cases (BLAS conventions):
 *   M == 0 or N == 0  -> DGEMM_OK, nothing is launched;
 *   K == 0 or alpha == 0 -> C = beta * C, A and B are never read; with
 *                           beta == 0 this writes zeros;
 *   beta == 0         -> C is never read, so NaN/Inf in it do not propagate.
 * Validation happens on the host before any launch; an invalid call writes
 *   nothing and launches nothing.  DGEMM_ERR_INVALID_ARG is returned for
 *   M, N or K < 0; a leading dimension smaller than its row length
 *   (lda < K; ldb < N for the NN calls, ldb < K for the TN calls; ldc < N);
 *   a NULL pointer for an operand that would be read or written.
 * DGEMM_ERR_UNSUPPORTED_DEVICE: the current device is not compute
 *   capability 10.3.
 * DGEMM_ERR_LAUNCH: the CUDA runtime reported an error at launch (the
 *   sticky error state of the context is not cleared).
 * Aliasing between C and A or B is not supported (results are undefined).
 * Any alignment is accepted; 16-byte aligned pointers and leading dimensions
 *   whose byte size is a multiple of 16 take the fastest kernels.
 * Indexing inside the kernels is 64-bit.
 */
#ifndef DGEMM_H
#define DGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_API_H__
struct CUstream_st;
typedef struct CUstream_st *cudaStream_t;
#endif

typedef enum {
    DGEMM_OK = 0,
    DGEMM_ERR_INVALID_ARG = 1,
    DGEMM_ERR_UNSUPPORTED_DEVICE = 2,
    DGEMM_ERR_LAUNCH = 3,
    DGEMM_ERR_TIMEOUT = 4,
    DGEMM_ERR_BOUNDS = 5  /* checked build only: a device-side bounds check failed */
} dgemm_status;

/*
 * gemm_f32 -- SGEMM on the FP32 pipes (CUDA cores, fused multiply-add in
 * single precision, round-to-nearest).
 *   M, N, K : problem size; A is M x K, B is K x N, C is M x N.
 *   alpha   : scale of the product;  beta: scale of the old C.
 *   A, lda  : device, float, row-major, element (m, k) at A[m*lda + k].
 *   B, ldb  : device, float, row-major, element (k, n) at B[k*ldb + n].
 *   C, ldc  : device, float, row-major, element (m, n) at C[m*ldc + n].
 *   stream  : CUDA stream (0 = legacy default stream).
 * Source: "SGEMM CUDA代码学习" (sections "第 1 步" to "第 4 步": block tile,
 * thread tile, bank-conflict-free staging, double buffering) and
 * "CUDA GEMM：从基础写法到工程优化" (sections 1 to 12, with alpha/beta).
 */
int gemm_f32(int64_t M, int64_t N, int64_t K, float alpha,
             const float *A, int64_t lda, const float *B, int64_t ldb,
             float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_tf32 -- same operation, signature and layouts as gemm_f32, but the
 * products run on the tensor cores in TF32 (each FP32 operand is reduced to
 * 1+8+10 bits inside the multiplier; the stored A and B are not modified),
 * with FP32 accumulation and an FP32 alpha/beta epilogue.
 * Large problems may take the stream-K schedule (see "Stream-K" above:
 * such calls are ordered across streams).
 * Source: "SGEMM CUDA代码学习", section "第 5 步" (TF32 tensor cores: a
 * 19-bit float, 1+8+10) and its WMMA TF32 multi-stage kernel.
 */
int gemm_tf32(int64_t M, int64_t N, int64_t K, float alpha,
              const float *A, int64_t lda, const float *B, int64_t ldb,
              float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_tf32_ws -- gemm_tf32 with a caller-provided scratch buffer for
 * operands that the tensor-memory-access (TMA) loads cannot describe: a base
 * that is not 16-byte aligned, or a leading dimension whose byte size is not
 * a multiple of 16 (e.g. lda = K = 4095).  Such an operand is first copied,
 * bit for bit, into the workspace with a padded pitch (A as M x
 * round_up(K, 4), B as K x round_up(N, 32) with zeros past column N), then
 * the TMA kernels run on the copy.  This replaces gemm_tf32's slower
 * element-wise loading path for those operands; results are the same as
 * gemm_tf32 on an aligned copy of the operands.
 *   workspace       : device buffer, 16-byte aligned, owned by the caller; it
 *                     must not overlap A, B or C and must stay untouched
 *                     until the stream has passed the call.  May be NULL
 *                     when gemm_tf32_workspace_bytes returns 0.
 *   workspace_bytes : its size in bytes.
 * Returns DGEMM_ERR_INVALID_ARG (nothing launched) when the workspace is
 * needed but is NULL, smaller than gemm_tf32_workspace_bytes() or not
 * 16-byte aligned; otherwise as gemm_tf32.  The call itself allocates
 * nothing.
 * Source: the operation of gemm_tf32; the repack is this library's way of
 * feeding the TMA loads ("SGEMM CUDA代码学习", "第 5 步", stages operands
 * through shared memory with asynchronous copies that need aligned
 * addresses as well).
 */
int gemm_tf32_ws(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 float beta, float *C, int64_t ldc,
                 void *workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * gemm_tf32_workspace_bytes -- workspace gemm_tf32_ws needs for these
 * operands: 0 when both A and B can be loaded as they are, else the bytes
 * of their padded copies; -1 for negative sizes, a leading dimension below
 * its row length, or sizes whose copies would not fit in 2^63 bytes.  Host
 * arithmetic only (no device access); the pointers are only looked at for
 * their alignment.
 */
int64_t gemm_tf32_workspace_bytes(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                  const float *B, int64_t ldb);

/*
 * gemm_f32_ws -- gemm_f32 with the workspace of gemm_tf32_ws (same layout,
 * same size: gemm_tf32_workspace_bytes).  When B's base or row pitch is not
 * a 16-byte multiple (e.g. ldb = N = 8193), B is first copied bit for bit
 * into the workspace with a padded pitch, so that the SIMT kernels load it
 * in 16-byte pieces (or by TMA) instead of 4-byte ones.  When A's base or
 * pitch is not a 16-byte multiple either and the problem has at least a
 * wave of output tiles, A is copied too, so that the TMA-fed kernel runs;
 * smaller problems (split-K) load A element by element and leave it in
 * place.  Results are the same as gemm_f32 on the same values.  Workspace
 * rules and errors as gemm_tf32_ws; the call allocates nothing.
 * Source: the operation of gemm_f32 ("SGEMM CUDA代码学习", "第 5 步":
 * 16-byte asynchronous copies need 16-byte aligned addresses).
 */
int gemm_f32_ws(int64_t M, int64_t N, int64_t K, float alpha,
                const float *A, int64_t lda, const float *B, int64_t ldb,
                float beta, float *C, int64_t ldc,
                void *workspace, int64_t workspace_bytes, cudaStream_t stream);

/* Size of the fixed scratch array behind gemm_tf32_noalloc (64 MiB). */
#define DGEMM_NOALLOC_SCRATCH_BYTES (64LL * 1024 * 1024)

/*
 * gemm_tf32_noalloc -- gemm_tf32_ws without a workspace argument, for callers
 * that cannot allocate device memory and so cannot provide one: for example
 * code running inside a host framework whose memory pool owns all of the
 * device's memory and refuses side allocations, or a latency-critical loop
 * in which an allocation (which may synchronise the device) is not
 * acceptable.  The caller still passes A, B and C as for gemm_tf32.
 * There is no counterpart in the pages: this is a property of the library,
 * not of the method.
 *   Scratch: a fixed array of DGEMM_NOALLOC_SCRATCH_BYTES in the library's
 *     device memory, which every GPU that loads the library holds until the
 *     process exits.  The call allocates nothing and frees nothing.
 *   Limit: operands whose padded copies need more than
 *     DGEMM_NOALLOC_SCRATCH_BYTES (see gemm_tf32_workspace_bytes) are
 *     rejected with DGEMM_ERR_INVALID_ARG and nothing is launched.  Operands
 *     that need no copy run as gemm_tf32_ws does, without touching it.
 *   Set-up: the first call on each device, made with that device current,
 *     looks up the array's device address; make that first call before any
 *     stream capture.  DGEMM_ERR_LAUNCH if the lookup fails.
 *   Sharing: every call uses the same array and each rewrites all of it that
 *     it reads, so no state carries over from one call to the next; two calls
 *     whose work overlaps on the GPU (different streams, or unordered calls
 *     from different host threads) race on the array and may corrupt each
 *     other's results.
 * Otherwise as gemm_tf32_ws.
 */
int gemm_tf32_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, float *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_f16_tn -- HGEMM in the TN layout: C = alpha * A * B^T + beta * C.
 *   A, lda  : device, IEEE binary16, M x K row-major, (m, k) at A[m*lda + k].
 *   B, ldb  : device, IEEE binary16, stored N x K row-major, so the logical
 *             B(k, n) is B[n*ldb + k] (ldb >= K).
 *   C, ldc  : device, IEEE binary16, M x N row-major.
 *   alpha, beta: float.
 * Products accumulate in FP32 on the tensor cores; alpha*acc + beta*C_old is
 * formed in FP32 and rounded once to binary16 (round to nearest even;
 * overflow gives +-Inf).
 * Source: "HGEMM SMEM Swizzle 代码学习" (FP16 TN tensor-core GEMM with a
 * swizzled shared-memory layout) and "Warp Specialization HGEMM" (producer /
 * consumer roles; section "6. B 的 RowMajor(K,N) 与 TN 布局").  The pages
 * accumulate in FP16; this library accumulates in FP32.
 */
int gemm_f16_tn(int64_t M, int64_t N, int64_t K, float alpha,
                const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                float beta, uint16_t *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_f16_nn -- HGEMM with every matrix row-major: C = alpha * A * B + beta * C.
 *   A, lda  : device, IEEE binary16, M x K row-major.
 *   B, ldb  : device, IEEE binary16, K x N row-major, (k, n) at B[k*ldb + n]
 *             (ldb >= N).
 *   C, ldc  : device, IEEE binary16, M x N row-major.
 * Arithmetic, rounding and special cases as gemm_f16_tn.
 * Source: "HGEMM SMEM Swizzle 代码学习", the kernel source's layout notes
 * ("NN: A/B/C all row major", next to the TN layout it implements).
 */
int gemm_f16_nn(int64_t M, int64_t N, int64_t K, float alpha,
                const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                float beta, uint16_t *C, int64_t ldc, cudaStream_t stream);

/*
 * gemm_bf16_tn / gemm_bf16_nn -- the same two layouts with bfloat16 A, B and
 * C (raw 16-bit patterns: 1 sign, 8 exponent, 7 fraction bits): products
 * accumulate in FP32 on the tensor cores; alpha*acc + beta*C_old is formed in
 * FP32 and rounded once to bfloat16 (nearest even).  TN: B stored N x K
 * (ldb >= K); NN: B stored K x N (ldb >= N).
 * Source: "SGEMM CUDA代码学习", section "第 5 步" (BF16 among the tensor-core
 * precisions, beside FP16 and TF32) with the layouts above.
 */
int gemm_bf16_tn(int64_t M, int64_t N, int64_t K, float alpha,
                 const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                 float beta, uint16_t *C, int64_t ldc, cudaStream_t stream);
int gemm_bf16_nn(int64_t M, int64_t N, int64_t K, float alpha,
                 const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                 float beta, uint16_t *C, int64_t ldc, cudaStream_t stream);

/* A static, NUL-terminated description of a dgemm_status value. */
const char *dgemm_status_string(int status);

/*
 * dgemm_device_status -- read (and, if clear != 0, reset) the current
 * device's kernel status word.  The tensor-core kernels and the TMA-fed
 * FP32 SIMT kernel bound every wait on an mbarrier; a wait that runs out
 * records DGEMM_ERR_TIMEOUT here and the kernel exits cleanly instead of
 * hanging.  This call synchronises the
 * device.  Returns DGEMM_OK when no kernel has recorded an error since the
 * last clear.  Source: none on the pages (they never check kernels).
 */
int dgemm_device_status(int clear);

/*
 * The checked build.  The library is also built as libdgemm_checked.so,
 * with the same ABI, compiled with -DDGEMM_CHECKED: every kernel then tests
 * the indices it computes -- shared-memory offsets (stage rings, swizzled
 * rows, epilogue boxes, split-K receive buffers), tile coordinates, global
 * rows and columns of A, B and C, the alignment of 16-byte accesses, TMEM
 * columns and stream-K workspace regions -- against the extents they must
 * stay inside.  A failed check skips the access it guards (no trap, nothing
 * out of bounds) and records DGEMM_ERR_BOUNDS in the device status (see
 * dgemm_device_status) and its site.  The checks cost time and are meant for
 * testing; in libdgemm.so they are compiled out.
 *
 * dgemm_check_site -- the site of the first failed check since the last
 * clear of the device status: (translation unit x 100000 + source line) of
 * the library's sources, units 1 sgemm_simt.cu, 2 sgemm_tma.cu,
 * 3 umma_gemm.cu, 4 scale_c.cu, 5 repack.cu; 0 if none failed, and always 0
 * in libdgemm.so.  Synchronises the device.  Source: none on the pages.
 */
int dgemm_check_site(void);

/*
 * dgemm_test_shrink_bounds -- TEST HOOK for the checked build.  The next
 * gemm_f32 launch of the TMA-fed SIMT kernel made by the calling host thread
 * checks its stores against M - rows rows of C instead of M, so that the
 * stores to the last `rows` rows fail their check: they are skipped and
 * reported (DGEMM_ERR_BOUNDS, a site in sgemm_tma.cu).  This shows that the
 * checks are live without any out-of-bounds access.  In libdgemm.so the
 * request is taken by the same launch and has no effect.  rows < 0 is
 * DGEMM_ERR_INVALID_ARG; otherwise returns DGEMM_OK.  Source: none on the
 * pages.
 */
int dgemm_test_shrink_bounds(int64_t rows);

/*
 * dgemm_test_inject_stall -- TEST HOOK, not for applications.  Arms a one-shot
 * fault for the next launch, made by the calling host thread, of a kernel
 * with bounded waits: a tensor-core kernel (gemm_tf32, the 16-bit calls) or
 * the TMA-fed FP32 SIMT kernel (gemm_f32 on aligned operands of at least a
 * wave of tiles).  That launch first waits on a barrier that nothing
 * arrives at (in the MMA issuer, or in every warp of the SIMT kernel), and
 * every wait of that launch is bounded by wait_limit_ns (0 means 1 ns)
 * instead of the default 4 s.  Calls that launch other kernels leave the
 * request armed.  The launch then ends by itself, with DGEMM_ERR_TIMEOUT in
 * the device status word (see dgemm_device_status) and C left unspecified;
 * the CUDA context stays usable.  Always returns DGEMM_OK.  Source: none on
 * the pages (they have no failure detection).
 */
int dgemm_test_inject_stall(uint64_t wait_limit_ns);

/*
 * dgemm_test_pair_units -- TEST HOOK, host computation only (no GPU needed).
 * Runs the CTA-pair kernels' work schedule, compiled for the host, for a 1-D
 * order of `tiles` tiles of num_kb K blocks on `pairs` pairs, with the first
 * sk_tiles tiles in the stream-K region (0, or at least `pairs`).  Writes the
 * units of pair `pair` in the order the pair runs them, 5 int64 each:
 * tile, first K block, end K block, init (starts from the previous pair's
 * partial), publish (leaves its partial for the next pair).  Writes at most
 * max_units units to out (caller-owned) and returns how many there are, or
 * -1 for arguments outside those ranges.  Source: none on the pages (their
 * kernels deal whole tiles).
 */
int64_t dgemm_test_pair_units(int64_t tiles, int64_t pairs, int64_t num_kb, int64_t sk_tiles, int64_t pair,
                              int64_t *out, int64_t max_units);

/*
 * dgemm_test_stream_k_tiles -- TEST HOOK, host only.  The stream-K region the
 * pair kernels would use for `tiles` tiles of num_kb K blocks on `pairs`
 * pairs: wide 1 (256 x 256 tiles) or 2 (256 x 512), mode 0 automatic, 1
 * never, 2 whenever the tiles outnumber the pairs.  Returns 0 (whole tiles),
 * pairs + tiles mod pairs, or -1 for an invalid wide or mode.
 */
int64_t dgemm_test_stream_k_tiles(int64_t tiles, int64_t pairs, int64_t num_kb, int wide, int mode);

/*
 * dgemm_test_choose_config -- TEST HOOK, host only.  The tile configuration
 * the tensor-core calls would choose automatically for an M x N x K problem
 * of `kind` (0 FP16 TN, 1 TF32, 2 BF16 TN, 3 FP16 NN, 4 BF16 NN) on a
 * device with sm_count SMs, assuming TMA-capable operands.  Writes the
 * variant (numbering of dgemm_tune_next), tile width and split / stream-K
 * mode; returns DGEMM_ERR_INVALID_ARG for non-positive sizes, sm_count < 2,
 * an unknown kind or a NULL output, else DGEMM_OK.  Small problems, whose
 * choice queries cluster occupancy on the current device, may choose
 * differently without a GPU.
 */
int dgemm_test_choose_config(int kind, int64_t M, int64_t N, int64_t K, int sm_count, int *variant, int *bn,
                             int *split);

/*
 * dgemm_tune_next -- TUNING HOOK.  Fixes the tile configuration of the next
 * tensor-core call (gemm_tf32, gemm_f16_*, gemm_bf16_*) made by the calling
 * host thread; one call only, after which the automatic choice resumes.
 *   variant 0: automatic (the default);
 *           1: CTA pair, 256 x 256 output tiles;
 *           2: one CTA per 128 x bn tile, persistent grid;
 *           3: split-K, `split` CTAs of a cluster per 128 x bn tile;
 *           4: not a variant (rejected with DGEMM_ERR_INVALID_ARG);
 *           5: CTA pair, 256 x 512 output tiles (one 512-column
 *              accumulator per CTA);
 *           6, 7: as 1 and 5 with the finer stage ring of the K-major
 *              16-bit calls (gemm_f16_tn, gemm_bf16_tn): 32-deep K stages
 *              under the 64-byte swizzle, twice as many in the same
 *              shared memory; other calls take 1 or 5 instead;
 *           8: CTA pair for small M, 128 x bn output tiles: one
 *              tcgen05.mma of M = 128 over the pair, each CTA loading 64
 *              rows of A and bn / 2 rows (columns, N-major) of B; one tile
 *              per pair, so only problems of at most one wave of pairs
 *              (the call chooses as usual otherwise).
 *   bn:    tile width for variants 2 and 3: 32..256 in steps of 32; the
 *          NN 16-bit calls need a multiple of 64.  For variant 8: 128, 192
 *          or 256 (the NN 16-bit calls: 128 or 256).  Ignored otherwise.
 *   split: 2..8 for variant 3 (lowered to the number of K blocks when K is
 *          shorter, so that every CTA has work); for variants 1, 5, 6 and 7
 *          the stream-K mode: 0 automatic, 1 whole tiles only, 2 cut the first
 *          P + (T mod P) of T tiles whenever they outnumber the P pairs;
 *          ignored otherwise.
 * Returns DGEMM_ERR_INVALID_ARG (and records nothing) for values outside
 * these ranges, else DGEMM_OK.  A configuration the next call cannot take
 * (operands that only the register-path kernel can load, or a bn that is not
 * a multiple of the call's step) is ignored, and the call chooses as usual;
 * dgemm_last_kernel() names what ran.  Results agree with the automatic
 * choice up to the order of the FP32 additions of split partials.  Source:
 * "如何优化一个 CUDA Matmul Kernel ... Worklog", section "Kernel 9:
 * Autotuning" (searching tile parameters per problem instead of fixing one).
 */
int dgemm_tune_next(int variant, int bn, int split);

/*
 * dgemm_last_kernel -- name of the kernel variant the last successful call
 * on this host thread launched ("" if none): for tests and the benchmark.
 */
const char *dgemm_last_kernel(void);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_H */
