/*
 * sgemm.h -- C ABI of the GB300 FP32 matrix-multiply library (libsgemm_gb300.so).
 *
 * The library computes the row-major FP32 product
 *
 *     C[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]        0 <= i < M, 0 <= j < N
 *
 * ("Micro Kernel 입문하기", §3, the GEMM formula held by the c_ij accumulators;
 *  "누산 개념을 Grid-Block-Warp-Thread 계층에 끼워넣기", §1-§2: one kernel launch
 *  completes all of C, each block owning a BM x BN tile of C, each warp a warp
 *  tile and each thread a TM x TN register tile accumulated over BK-deep
 *  shared-memory slices; "Register/Shared Memory Tiling", 동작 원리.)
 *
 * Layout.  Every matrix is row-major with a leading dimension counted in
 * elements: A[i,k] = A[i*lda + k], B[k,j] = B[k*ldb + j], C[i,j] = C[i*ldc + j]
 * (the pages' `A[gm * p.lda + gk]` and `C[m * p.ldd + n]`, "기존 작성한 GE_v2 의
 * regemm 타일드 커널의 1:1 매핑, gemm_tiled_test 작성", §3 and §6).
 *
 * Semantics.  C is overwritten (beta = 0, alpha = 1).  Elements of C outside the
 * M x N region, including the padding between rows when ldc > N, are never
 * written; elements of A and B outside their logical extents are never read
 * (the tile loads substitute zeros there, ibid. §3 "boundary check 후 0-padding").
 * K == 0 writes zeros to C (the empty sum).  M == 0 or N == 0 is a no-op.
 * M, N and K may each be at most 2^30 (the kernels keep tile bounds in 32-bit
 * integers; element offsets are 64-bit); larger ones return SGEMM_ERR_UNSUPPORTED.
 *
 * Memory.  A, B and C are DEVICE pointers owned by the caller.  C must not
 * overlap A or B.  Any alignment of pointers and leading dimensions is accepted;
 * 16-byte-aligned operands with leading dimensions that are multiples of 4 take
 * the vectorised kernels, others a 4-byte-granular variant.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 * call is asynchronous on that stream and does not synchronise the host.
 *
 * Threads.  Entry points may be called from several host threads at once.  Calls
 * that use the library-owned workspace of one (device, stream) hold its lock from
 * the workspace lookup until their launches are enqueued, so a call that grows
 * it never frees a buffer another call is about to launch with; calls on other
 * streams do not wait for each other.  sgemm_shutdown is the exception: it must
 * not run concurrently with any other call.
 *
 * Errors.  Every entry point returns an sgemm_status and never aborts the
 * process.  Invalid arguments are rejected before anything is launched.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SGEMM_API __attribute__((visibility("default")))
#else
#define SGEMM_API
#endif

struct CUstream_st;                       /* cudaStream_t == struct CUstream_st* */
typedef struct CUstream_st* sgemm_stream_t;

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = -1,   /* bad size, leading dimension, null or aliased pointer */
    SGEMM_ERR_ALIGNMENT = -2,     /* reserved: misalignment selects another kernel instead */
    SGEMM_ERR_LAUNCH = -3,        /* a CUDA call failed (message: sgemm_last_error()) */
    SGEMM_ERR_UNSUPPORTED = -4,   /* no device, wrong architecture, unknown kernel id,
                                     M, N or K above 2^30 */
    SGEMM_ERR_TIMEOUT = -5,       /* a bounded device-side wait gave up */
    SGEMM_ERR_WORKSPACE = -6      /* caller workspace too small, or allocation failed */
} sgemm_status;

/* One entry of the tile table, as chosen for a problem.  `kernel_id` indexes the
 * table (0 .. sgemm_num_kernels()-1).  `split_k` is the number of CTAs that share
 * the K range of a split tile (1 = data-parallel only); `grid` the CTAs launched
 * (a persistent grid); `sk_tiles` the tiles finished by several CTAs. */
typedef struct {
    int bm, bn, bk;        /* block tile of C and depth of one shared-memory slice */
    int wm, wn;            /* warp tile */
    int tm, tn;            /* register tile of one thread */
    int stages;            /* shared-memory pipeline depth */
    int threads;           /* threads per CTA */
    int smem_bytes;        /* dynamic shared memory per CTA */
    int split_k;           /* max CTAs sharing one tile's K range (1 = none) */
    int kernel_id;         /* index into the tile table */
    int vec;               /* 4: 16-byte global loads; 1: 4-byte loads (any alignment) */
    int grid;              /* CTAs launched */
    int tiles;             /* BM x BN tiles of C */
    int sk_tiles;          /* tiles completed by more than one CTA (stream-K) */
    int ctas_per_sm;       /* resident CTAs per SM for this kernel */
    int fma2;              /* 1: packed fma.rn.f32x2 micro-kernel */
    int packed;            /* sgemm_run copies A (bit 0) / B (bit 1) to aligned buffers first */
    int sk_gap;            /* stream-K: k-slices of store time counted between split tiles
                              when the K ranges are shared out (0: equal ranges) */
    int cluster;           /* cluster split: CTAs per tile, one thread-block cluster each,
                              summing their partial tiles in distributed shared memory in
                              a fixed order, in the same launch (0: not used) */
} sgemm_config;

/* C = A.B on `stream`.  One kernel launch, plus a second, short reduction launch
 * when the schedule splits the K range of some tiles between CTAs (stream-K);
 * the partial tiles then go to a library-owned device workspace (allocated on
 * first use per device and stream with the stream-ordered allocator, grown when
 * a larger one is needed, freed by sgemm_shutdown).  Problems of less than one
 * resident wave of tiles may instead split every tile's K range over a
 * thread-block cluster of 2, 4 or 8 CTAs that sum their partial tiles in
 * distributed shared memory, in k order, inside the one launch; that needs no
 * workspace (sgemm_query_config reports it as `cluster`).  Problems with K >= 768
 * and M*N*K >= 5e8 whose A or B rows are not 16-byte aligned are first copied row
 * by row into aligned buffers in that workspace (one more launch per copied operand),
 * so they run on the 16-byte / TMA kernels (the copy moves values, not sums: the
 * results are those of the aligned kernels on aligned operands; they can differ
 * from the 4-byte-load kernels' in rounding, as any two tilings can, and stay
 * within the same bound).  The first call that needs a workspace must not be
 * made while the stream is being captured into a CUDA graph.  One workspace is
 * kept for every (device, stream handle) that needed one, until sgemm_shutdown;
 * a program that cycles through many short-lived streams is better served by
 * sgemm_run_ws or sgemm_run_noalloc.  The product kernel is launched as a
 * programmatic dependent of the stream's previous kernel: its set-up may overlap
 * that kernel's tail, and it waits for that kernel to complete before reading or
 * writing global memory, so stream order holds as for a plain launch
 * (SGEMM_PDL=0 launches it plainly). */
SGEMM_API int sgemm_run(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
              float* C, int ldc, sgemm_stream_t stream);

/* Scaled form: C = alpha * A.B + beta * C, with the BLAS conventions: when
 * beta == 0, C is only written (its old contents, NaN included, are ignored);
 * when alpha == 0 or K == 0, A and B are not read and C = beta * C.  The plain
 * entry points are this with alpha = 1, beta = 0.  ("기존 작성한 GE_v2 의 regemm
 * 타일드 커널의 1:1 매핑, gemm_tiled_test 작성" names the GE_v2 kernel's epilogue,
 * which its test kernel removes; the scaling rule itself is the BLAS one.)
 * The scaled value is fmaf(alpha, acc, beta * c) per element.  kernel_id = -1 and
 * schedule = 0 select automatically; other values force a tile-table entry and
 * schedule as for sgemm_run_with.  alpha or beta NaN -> SGEMM_ERR_INVALID_ARG. */
SGEMM_API int sgemm_run_ex(int M, int N, int K, float alpha, const float* A, int lda,
                           const float* B, int ldb, float beta, float* C, int ldc,
                           int kernel_id, int schedule, sgemm_stream_t stream);

/* As sgemm_run, with a caller-owned device workspace of `ws_bytes` bytes (at least
 * sgemm_workspace_size() for the same arguments, 16-byte aligned; may be NULL
 * when that size is 0).  The library allocates nothing on this path.  The
 * workspace needs no initialisation; it must stay untouched by other work while
 * the call runs and must not be shared by calls that can overlap on the GPU.
 * Returns SGEMM_ERR_WORKSPACE if it is missing or too small. */
SGEMM_API int sgemm_run_ws(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                 float* C, int ldc, void* ws, size_t ws_bytes, sgemm_stream_t stream);

/* Size of the static scratch array sgemm_run_noalloc uses (40 MiB). */
#define SGEMM_NOALLOC_SCRATCH_BYTES (40u << 20)

/* As sgemm_run, but the library allocates no device memory at all; for callers
 * that cannot let a library call cudaMalloc (it can synchronise the device and
 * take unbounded time on a latency-critical path, and some processes reserve
 * their whole device memory budget up front).  The source pages have no
 * counterpart to this entry point: it exists only for such callers.
 *
 * When the schedule splits tiles between CTAs through a workspace (stream-K),
 * the partial tiles go to one static __device__ array of
 * SGEMM_NOALLOC_SCRATCH_BYTES compiled into the library; problems whose tiles
 * are split inside thread-block clusters, or not split at all, use no scratch.
 * A problem that would need more scratch than the array holds is rejected with
 * SGEMM_ERR_WORKSPACE and a message in sgemm_last_error(); nothing is launched.
 *
 * Set-up: the first call on a device that needs the scratch looks up the
 * array's device address (with that device current).  Under CUDA's default lazy
 * module loading that lookup is also what loads the library module holding the
 * array, so that first call reserves SGEMM_NOALLOC_SCRATCH_BYTES of device
 * memory (as the first launch of any kernel loads that kernel's code); from
 * then on the device holds the array until the process exits, and later calls
 * allocate nothing.  Make that first call at set-up time, before any stream
 * capture begins and before the device's memory budget is fixed.  The address
 * is kept per device index for the primary context and looked up again after
 * sgemm_shutdown.
 *
 * All calls on a device share the array, so calls that can overlap on the GPU
 * (e.g. on different streams without ordering between them) race and must not
 * be issued; calls ordered on one stream are fine.  Like sgemm_run_ws (it is
 * that call with the static array as workspace), it never copies misaligned
 * operands to aligned buffers first, so for such operands it may run another
 * tile-table entry than sgemm_run and round differently, within the same bound.
 * A, B, C and `stream` are as for sgemm_run. */
SGEMM_API int sgemm_run_noalloc(int M, int N, int K, const float* A, int lda, const float* B,
                                int ldb, float* C, int ldc, sgemm_stream_t stream);

/* Bytes of workspace sgemm_run_ws needs for these arguments on the current
 * device (0 if none).  The pointers matter only through their alignment, which
 * selects the tile-table entry; NULL assumes a 16-byte-aligned operand, so pass
 * the real pointers when they may be misaligned (sgemm_run_ws rejects a workspace
 * that turns out too small with SGEMM_ERR_WORKSPACE; it never overruns it).
 * Returns SGEMM_ERR_INVALID_ARG for a negative size, a leading dimension below
 * its row width or a NULL out_bytes, and SGEMM_ERR_UNSUPPORTED when the current
 * device is not an sm_103 GPU. */
SGEMM_API int sgemm_workspace_size(int M, int N, int K, int lda, int ldb, int ldc,
                         const float* A, const float* B, const float* C, size_t* out_bytes);

/* As sgemm_run, forcing tile-table entry `kernel_id` (for tests and tuning) and a
 * schedule: `schedule` 0 = automatic, 1 = data-parallel only, 2 = stream-K on the
 * last partial wave whenever it has at least one k-tile per CTA, 3 = every tile
 * split over a cluster of the largest power of two up to 8 CTAs that leaves each
 * a k-tile (the TMA-fed entries, which cannot sum in a cluster, plan as for 0).
 * Returns
 * SGEMM_ERR_UNSUPPORTED if that entry cannot serve these operands (e.g. a
 * 16-byte-load entry for unaligned operands). */
SGEMM_API int sgemm_run_with(int M, int N, int K, const float* A, int lda, const float* B, int ldb,
                   float* C, int ldc, int kernel_id, int schedule, sgemm_stream_t stream);

/* The configuration sgemm_run would use for these arguments on the current
 * device.  Pointers only matter through their alignment; pass NULL to assume
 * 16-byte-aligned operands. */
SGEMM_API int sgemm_query_config(int M, int N, int K, int lda, int ldb, int ldc,
                       const float* A, const float* B, const float* C, sgemm_config* out);

/* Transposed operands, BLAS style:  C = alpha * op(A) . op(B) + beta * C  with
 * op(A) M x K and op(B) K x N.  transa == 0: A is stored M x K row-major
 * (lda >= K); transa == 1: A is stored K x M row-major (lda >= M) and
 * op(A) = A^T.  transb == 0: B is stored K x N (ldb >= N); transb == 1: B is
 * stored N x K (ldb >= K) and op(B) = B^T.  C is M x N row-major (ldc >= N).
 * Row-major with a transposed operand is the pages' product on op(A), op(B)
 * ("Register/Shared Memory Tiling", 관련 개념: the tile hierarchy does not depend
 * on which operand is stored k-major).  A transposed operand is first
 * transposed into a 16-byte-aligned row-major buffer of the library workspace
 * (an HBM-bound pass of 8 bytes per element), then the product runs on that
 * buffer exactly as sgemm_run_ex would.  Device pointers, asynchronous on
 * `stream`.  Errors: as sgemm_run_ex,
 * plus SGEMM_ERR_INVALID_ARG for transa or transb other than 0 or 1, ld values
 * below the stored row widths, or C overlapping the stored A or B. */
SGEMM_API int sgemm_run_op(int transa, int transb, int M, int N, int K, float alpha,
                           const float* A, int lda, const float* B, int ldb, float beta, float* C,
                           int ldc, sgemm_stream_t stream);

/* Host-buffer convenience for end-to-end use: copies A and B from host memory
 * (pinned for full speed) into the caller's device buffers dA, dB (row-major,
 * leading dimensions lda, ldb), computes C = A.B into dC (leading dimension ldc)
 * and copies C back to hC.  The work is ordered after everything already queued
 * on `stream`, and `stream` waits for all of it, so it behaves as if issued on
 * `stream`; inside, it runs on three library-owned streams of the current device
 * (created on first use, destroyed by sgemm_shutdown) so that copies overlap the
 * product: C is computed in row panels; the first panel's product is summed over
 * k-chunks (beta = 1 after the first) as its chunk of A and B arrives, the other
 * panels start once their rows of A are in, and each finished panel is copied
 * back while the next one is computed.  Rounding can differ from sgemm_run's by
 * that chunking; the error bound is the same.  A problem planned as one panel
 * (fewer than 5e8 multiply-adds) has nothing to overlap: its copies and product
 * are queued on `stream` itself.  The call returns when the work is
 * queued; synchronise
 * `stream` before reading hC.  Calls from several host threads are serialised
 * while they queue.  Errors: as sgemm_run, plus SGEMM_ERR_INVALID_ARG for a null
 * device buffer with a non-empty extent and SGEMM_ERR_LAUNCH for a failed copy;
 * after an error, `stream` is still ordered after whatever part was queued. */
SGEMM_API int sgemm_run_host(int M, int N, int K, const float* hA, int lda, const float* hB, int ldb,
                   float* hC, int ldc, float* dA, float* dB, float* dC,
                   sgemm_stream_t stream);

/* Most row panels (and k-chunks of the first panel) sgemm_run_host splits into. */
#define SGEMM_HOST_MAX_PANELS 16

/* Host-only view of sgemm_run_host's plan (no GPU needed): the number of row
 * panels of C in *n_panels, their heights in rows[0 .. *n_panels - 1] (rows may
 * be NULL; else it holds SGEMM_HOST_MAX_PANELS ints) and the depth of the first
 * panel's k-chunks in *k_chunk (K when it is not chunked, 0 for K == 0; may be
 * NULL).  The panels cover M in order, every one but the last a multiple of 256
 * rows.  The tuning variables SGEMM_HOST_SPLIT, SGEMM_HOST_PANELS and
 * SGEMM_HOST_KCHUNKS are honoured as in sgemm_run_host.  Returns
 * SGEMM_ERR_INVALID_ARG for M or N <= 0, K < 0 or a NULL n_panels. */
SGEMM_API int sgemm_host_plan_check(int M, int N, int K, int* n_panels, int* rows, int* k_chunk);

/* 3xTF32 tensor-core variant (tcgen05, TMEM, TMA): C = alpha * A.B + beta * C with
 * each operand split into two TF32 numbers, x = hi + lo, and
 * A.B ~= Ahi.Bhi + Ahi.Blo + Alo.Bhi accumulated in fp32 in tensor memory
 * ("Register/Shared Memory Tiling", 관련 개념 / 장단점: pairing the tile
 * hierarchy with tensor-core MMA).  Accuracy is FP32-class but not the CUDA-core
 * path's: the tolerance is max|C - C_ref| <= 1e-5 * K * max|A| * max|B|.  Inf and
 * NaN inputs are not supported (the split turns Inf into NaN).  The split
 * operands go to a workspace of sgemm_tf32x3_workspace_size() bytes: the caller's
 * `ws` (16-byte aligned, ws_bytes large enough) or, when ws is NULL, the library's
 * per-stream workspace (allocated on first use).  The workspace also holds the
 * partial tiles when the schedule splits tiles between CTAs.  Launches the
 * operand split, the GEMM and, for split tiles, a deterministic reduction.  Any
 * alignment of A, B, C and any leading dimensions.  When A's rows are 16-byte
 * aligned (A 16-byte aligned, lda % 4 == 0) the GEMM reads A itself as the hi
 * part (the tensor core reads fp32 as TF32 by dropping the 13 low mantissa bits,
 * which is the split's hi) and the split writes only the lo part of A; the
 * results are the same bit for bit.  SGEMM_TF32X3_SPLIT_A=1 writes both parts.
 * Bounded device-side waits that give up set a flag read by sgemm_device_status(). */
SGEMM_API int sgemm_tf32x3_run(int M, int N, int K, const float* A, int lda, const float* B,
                               int ldb, float* C, int ldc, sgemm_stream_t stream);
SGEMM_API int sgemm_tf32x3_run_ex(int M, int N, int K, float alpha, const float* A, int lda,
                                  const float* B, int ldb, float beta, float* C, int ldc,
                                  void* ws, size_t ws_bytes, sgemm_stream_t stream);
SGEMM_API int sgemm_tf32x3_workspace_size(int M, int N, int K, size_t* out_bytes);

/* The configuration sgemm_tf32x3_run_ex would use for M x N x K on the current
 * device: bm x bn output tiles (bn 128 or 256, chosen per problem), bk = 32-deep
 * k-blocks, stages, threads, shared memory, the persistent grid, the tile count,
 * the tiles split by k-blocks over several CTAs (sk_tiles; their partials are
 * summed by a second, deterministic kernel) and the most CTAs sharing one
 * (split_k).  kernel_id is -1 (not a tile-table entry).  Errors:
 * SGEMM_ERR_INVALID_ARG for a null `out` or a non-positive size. */
SGEMM_API int sgemm_tf32x3_query_config(int M, int N, int K, sgemm_config* out);

/* The two steps of sgemm_tf32x3_run_ex, for callers that reuse operands or time
 * the steps apart.  _prepare writes the TF32 hi/lo parts of A (M x K) and the
 * transposed parts of B (K x N) into `ws` (caller-owned, 16-byte aligned, at
 * least sgemm_tf32x3_workspace_size(M, N, K) bytes); _multiply then computes
 * C = alpha * A.B + beta * C from that workspace only.  Both are asynchronous
 * on `stream`; the workspace must not change between them. */
SGEMM_API int sgemm_tf32x3_prepare(int M, int N, int K, const float* A, int lda, const float* B,
                                   int ldb, void* ws, size_t ws_bytes, sgemm_stream_t stream);
SGEMM_API int sgemm_tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C,
                                    int ldc, const void* ws, size_t ws_bytes,
                                    sgemm_stream_t stream);

/* Synchronous: reads and clears the device flag that a bounded wait in a
 * tensor-core kernel sets when it gives up; returns SGEMM_ERR_TIMEOUT if it was
 * set, SGEMM_OK otherwise.  Call after synchronising the work in question. */
SGEMM_API int sgemm_device_status(void);

/* Failure-detection self-test (synchronous): launches one CTA that waits, with
 * the same time-bounded mbarrier wait the TMA-fed kernels use but a limit of
 * `limit_ms` (1..10000), on a barrier that nothing completes.  The wait must
 * give up by itself and record the timeout; returns SGEMM_ERR_TIMEOUT when it
 * did (the expected result, read and cleared through sgemm_device_status), and
 * SGEMM_OK if the wait was never recorded.  The context stays usable. */
SGEMM_API int sgemm_selftest_bounded_wait(int limit_ms);

/* Host-only check of the persistent / stream-K schedule (no GPU needed): plans
 * M x N x K for tile-table entry `kernel_id` as if `sms` SMs each held
 * `ctas_per_sm` CTAs, then walks every CTA's list of k-slices the way the kernel
 * does.  Returns SGEMM_OK if every (tile, k-slice) is computed exactly once and
 * every split tile's partial slots and contributor count are consistent, else
 * SGEMM_ERR_INVALID_ARG with the reason in sgemm_last_error().  `out` (may be
 * NULL) receives the planned configuration. */
SGEMM_API int sgemm_schedule_check(int M, int N, int K, int kernel_id, int sms, int ctas_per_sm,
                                   int schedule, sgemm_config* out);

/* Host-only view of the per-shape tile table (no GPU needed): the entry that
 * sgemm_run picks for an M x N x K product with leading dimensions lda, ldb (in
 * floats) on a GPU with `sms` SMs.  `a_offset` and `b_offset` (0..3) place the
 * start of A and B that many floats past a 16-byte boundary.  As in sgemm_run,
 * a large product with a misaligned operand is planned on its aligned packed
 * copy; `packed` (may be NULL) receives 1 if A would be packed, 2 if B, 3 for
 * both.  SGEMM_FORCE_KERNEL is not consulted.  Returns SGEMM_ERR_INVALID_ARG for
 * M, N or K <= 0, lda < K, ldb < N, sms <= 0, an offset outside 0..3 or a NULL
 * kernel_id. */
SGEMM_API int sgemm_choose_check(int M, int N, int K, int lda, int ldb, int a_offset,
                                 int b_offset, int sms, int* kernel_id, int* packed);

/* Number of entries in the tile table, and entry `kernel_id`'s static shape
 * (grid, tiles, sk_tiles and split_k are left 0). */
SGEMM_API int sgemm_num_kernels(void);
SGEMM_API int sgemm_kernel_info(int kernel_id, sgemm_config* out);

/* Name of tile-table entry `kernel_id` ("" if out of range; static storage). */
SGEMM_API const char* sgemm_kernel_name(int kernel_id);

/* Human-readable name of a status code (static storage). */
SGEMM_API const char* sgemm_status_string(int status);

/* Text of the last CUDA error seen by this thread (static per-thread storage). */
SGEMM_API const char* sgemm_last_error(void);

/* Kernels this library has launched in this process (for launch accounting). */
SGEMM_API uint64_t sgemm_launch_count(void);

/* Frees the library-owned workspaces on every device, destroys the host-buffer
 * entry point's streams and events, and forgets the per-device state the library
 * keeps (kernel attributes set in the device's context, the allocation-free
 * entry's scratch addresses).  The library can be used again afterwards,
 * including after cudaDeviceReset: that state is set up again on first use.  Not
 * thread-safe with any concurrent call into the library. */
SGEMM_API int sgemm_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
