/*
 * sgemm.h - C ABI of the GB300 (sm_103a) single-precision matrix product library.
 *
 * The operation is the one stated in "LeetGPU | 02_Matrix_Multiplication", sections
 * "Problem Description" and "Constraints", and in "CUDA 学习笔记 Matrix
 * Multiplication", section "1. 题目含义":
 *
 *     C = A . B,   C[m][k] = sum over n = 0 .. N-1 of A[m][n] * B[n][k]
 *
 * A is M x N, B is N x K and C is M x K. All three are dense row-major float32 with no
 * padding: A[m*N + n], B[n*K + k], C[m*K + k]. The reduction runs over N.
 * 1 <= M, N, K <= 8192.
 *
 * Common rules for every entry point below:
 *  - Pointers named A, B, C are DEVICE pointers (cudaMalloc, cudaMallocAsync or a
 *    PyTorch CUDA tensor's storage) on the current CUDA device. The caller owns them;
 *    the library never frees or keeps them past the call.
 *  - No alignment is required. 16-byte aligned pointers with N % 4 == 0 and K % 4 == 0
 *    take the vectorised and TMA paths; anything else takes loaders that read 4-byte
 *    elements, with the same results.
 *  - C is overwritten; its old contents are ignored (no alpha/beta). Every element
 *    of C is written.
 *  - C must not overlap A or B. A and B may overlap each other.
 *  - Inputs are assumed finite. (With SGEMM_MODE_FP32_3XTF32 an infinite input gives
 *    NaN outputs, because the split x - hi(x) of an infinity is NaN.)
 *  - Work is enqueued on the given stream and the call returns without waiting,
 *    except solve_host (which waits) and the query calls documented as waiting.
 *  - Argument errors are detected on the host before anything is enqueued.
 *  - Status codes: 0 on success, a negative SGEMM_ERR_* value otherwise.
 *  - Streams are passed as void* holding a cudaStream_t; NULL (0) is the legacy
 *    default stream.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

/* Only the functions below are exported from the shared library. */
#if defined(SGEMM_BUILD) && defined(__GNUC__)
#define SGEMM_API __attribute__((visibility("default")))
#else
#define SGEMM_API
#endif

/* ---- status codes ---- */
#define SGEMM_OK 0
#define SGEMM_ERR_ARG (-1)         /* dimension outside [1, 8192], null pointer, bad mode */
#define SGEMM_ERR_OVERLAP (-2)     /* C overlaps A or B */
#define SGEMM_ERR_CUDA (-3)        /* a CUDA runtime call failed (launch, copy, allocation) */
#define SGEMM_ERR_NO_DEVICE (-4)   /* no CUDA device, or the current device is not sm_103 */
#define SGEMM_ERR_TIMEOUT (-5)     /* a bounded wait inside a kernel gave up (device error word) */
#define SGEMM_ERR_UNSUPPORTED (-6) /* the mode cannot serve this shape */

/* ---- arithmetic modes ----
 * SGEMM_MODE_FP32: FP32-accurate. Contract: |C - C_exact| <= 1e-5 * (|A|.|B|)[m][k]
 *   elementwise on the workloads' inputs (uniform and normal entries), and bit-exact
 *   when every partial sum is an exactly representable float (for instance
 *   integer-valued inputs with |value| <= 2048 and partial sums below 2^24). The
 *   library picks the fastest kernel that meets this for the shape: the streaming
 *   kernels for M == 1 or K == 1, the short-reduction kernel for N <= 4, the
 *   CUDA-core kernel when M*N*K <= 2^22, or <= 2^27 with N <= 1024 (one launch, no
 *   workspace), and the segmented 3xTF32 tensor-core kernel otherwise.
 * SGEMM_MODE_TF32: the explicit 1xTF32 tensor-core product of "LeetGPU |
 *   02_Matrix_Multiplication", section "V5: WMMA TF32 Tensor Core Kernel": each input
 *   is rounded to TF32 (10 explicit mantissa bits, round to nearest with ties away
 *   from zero) and products are accumulated in FP32. Contract: |C - C_exact| <=
 *   2e-3 * (|A|.|B|)[m][k]; bit-exact on integer inputs with |value| <= 2048.
 *   Shapes with M == 1, K == 1 or N <= 4 use the FP32 streaming kernels, which are
 *   bound by memory traffic there and meet the tighter FP32 contract.
 * SGEMM_MODE_FP32_SIMT: force the CUDA-core FFMA kernel (FP32 contract; bit-exact
 *   on integer inputs whose partial sums stay below 2^24).
 * SGEMM_MODE_FP32_3XTF32: force the split-precision tensor-core kernel: each input is
 *   split as x = hi + lo with hi = x truncated to TF32 and lo = x - hi rounded to TF32,
 *   three TF32 products per term (lo.hi, hi.lo, hi.hi) are accumulated in short
 *   tensor-core segments that are summed in FP32 registers (FP32 contract).
 * SGEMM_MODE_3XFP16_SCALED: split-precision on the 16-bit tensor path, which multiplies
 *   twice as many elements per clock: each row of A and each block of 128 columns of B
 *   is first scaled by a power of two that puts its largest magnitude in [2^14, 2^15); each
 *   scaled input is split as hi = x rounded to FP16 and lo = x - hi rounded to FP16 (22
 *   significant bits in all); three FP16 products per term are accumulated as in
 *   3xTF32, and the epilogue undoes the two scales exactly. An element far below its
 *   row's (block's) largest magnitude keeps fewer bits, because its lo piece falls
 *   below FP16's normal range. Contract: |C - C_exact| <= 1e-5 * (|A|.|B|)[m][k] +
 *   2^-37 * (max_n |A[m][n]| * sum_n |B[n][k]| + sum_n |A[m][n]| * maxB(k)), maxB(k)
 *   the largest |B| in the 128-column block of k; the second term matters only when a
 *   few terms far below their row's or block's largest make up most of
 *   (|A|.|B|)[m][k] (a product with the identity, say): on the
 *   workloads' uniform, normal and integer inputs the first alone holds. Bit-exact on
 *   integer inputs with |value| <= 2048 whose partial sums stay below 2^24. Every shape
 *   runs the tensor-core kernel. This mode does NOT meet the FP32 contract above for
 *   every finite input (A times the identity, with elements of a row spread over more
 *   than 2^17, misses it), so it is not FP32 and is never chosen by SGEMM_MODE_FP32. */
#define SGEMM_MODE_FP32 0
#define SGEMM_MODE_TF32 1
#define SGEMM_MODE_FP32_SIMT 2
#define SGEMM_MODE_FP32_3XTF32 3
#define SGEMM_MODE_3XFP16_SCALED 4

/* ---- kernel identifiers returned by sgemm_plan ---- */
#define SGEMM_KERNEL_SIMT 1      /* CUDA-core FFMA GEMM, any shape */
#define SGEMM_KERNEL_GEVM 2      /* M == 1: stream B, deterministic split-N reduction */
#define SGEMM_KERNEL_GEMV 3      /* K == 1: stream A, one warp per output row */
#define SGEMM_KERNEL_TC_1XTF32 4 /* tcgen05 TF32 GEMM, one product per term */
#define SGEMM_KERNEL_TC_3XTF32 5 /* tcgen05 TF32 GEMM, three products per term */
#define SGEMM_KERNEL_SMALLN 6    /* N <= 4: FP32 FMA, bound by writing C once */
#define SGEMM_KERNEL_TC_3XFP16 7 /* tcgen05 FP16 GEMM, three products of scaled pieces */

/* Rate probes for sgemm_peak_probe */
#define SGEMM_PROBE_FFMA 0     /* scalar FP32 fused multiply-add (CUDA cores) */
#define SGEMM_PROBE_FFMA2 1    /* packed FP32 FMA, two lanes per instruction (CUDA cores) */
#define SGEMM_PROBE_TF32_MMA 2 /* tcgen05 kind::tf32 pair MMA, M=256 N=256 K=8 */
#define SGEMM_PROBE_F16_MMA 3  /* tcgen05 kind::f16 pair MMA, FP16 operands, M=256 N=256 K=16 */

/*
 * solve - the problem statement's entry point, signature unchanged from "LeetGPU |
 * 02_Matrix_Multiplication", sections "Implementation Requirements" and "V0 ...
 * Solution": C = A . B in SGEMM_MODE_FP32.
 *
 * A (M x N), B (N x K), C (M x K): device pointers, row-major float32. Enqueues on
 * the calling thread's stream (sgemm_set_stream; default: legacy default stream) and
 * returns without waiting. It returns void, like the pages' version; the status is
 * kept for sgemm_last_status(), and launch failures also show in cudaGetLastError().
 */
SGEMM_API void solve(const float* A, const float* B, float* C, int M, int N, int K);

/*
 * solve_ex - C = A . B with an explicit arithmetic mode (SGEMM_MODE_*) on an explicit
 * stream (a cudaStream_t, NULL for the legacy default stream). Arguments as for solve.
 * Returns SGEMM_OK or a negative SGEMM_ERR_* code; on an argument error nothing is
 * enqueued and C is untouched. Temporary workspace (TF32 operand planes, split-N
 * partial sums) comes from a library-owned stream-ordered memory pool on the same
 * stream, so stream order is kept and no host synchronisation happens. Everything the
 * call enqueues is stream-ordered, so it may be captured into a CUDA graph and replayed
 * (the replay reads whatever A and B then hold); make one call of the same kind outside
 * capture first, which loads the kernels and sets their attributes.
 */
SGEMM_API int solve_ex(const float* A, const float* B, float* C, int M, int N, int K, int mode,
             void* stream);

/*
 * solve_host - C = A . B for HOST arrays: copies A and B to the device, runs solve_ex
 * on `stream`, copies C back and waits for the stream. hA (M*N floats), hB (N*K
 * floats) and hC (M*K floats) are host pointers owned by the caller; page-locked
 * memory gives full copy speed. Device buffers come from the library's pool and are
 * returned to it before the call ends. Returns SGEMM_OK or SGEMM_ERR_*. This is the
 * round trip (upload A, upload B, kernel, download C) measured in "分块计算与矩阵乘法",
 * section "结果与测量边界". For tensor-core products with M >= 2048 the round trip is
 * pipelined: B is uploaded first, then A's rows are uploaded, split, multiplied and C's
 * rows downloaded in chunks of 1024 rows on the library's own copy and split streams,
 * overlapping each other; `stream` carries the GEMMs.
 */
SGEMM_API int solve_host(const float* hA, const float* hB, float* hC, int M, int N, int K,
                         int mode, void* stream);

/* sgemm_set_stream - stream used by solve() on the calling thread (thread-local).
 * Returns SGEMM_OK. */
SGEMM_API int sgemm_set_stream(void* stream);

/* sgemm_last_status - status of the calling thread's most recent solve() call. */
SGEMM_API int sgemm_last_status(void);

/* sgemm_status_string - static English text for a status code (never NULL). */
SGEMM_API const char* sgemm_status_string(int status);

/*
 * sgemm_device_error - waits for `stream`, then reads and clears the current device's
 * error word. Kernels set it when one of their bounded waits gives up instead of
 * hanging. Returns SGEMM_OK, SGEMM_ERR_TIMEOUT, or SGEMM_ERR_CUDA if the read failed.
 */
SGEMM_API int sgemm_device_error(void* stream);

/*
 * sgemm_plan - host-only dispatch query: the SGEMM_KERNEL_* that solve_ex would launch
 * for this shape, mode and pointer alignment (aligned = 1 when A, B and C are 16-byte
 * aligned), assuming an sm_103 device. Writes the output tile count to *tiles when
 * tiles is not NULL. Touches no device. Returns a kernel id (> 0) or SGEMM_ERR_*.
 */
SGEMM_API int sgemm_plan(int M, int N, int K, int mode, int aligned, int* tiles);

/*
 * sgemm_plan_units - host-only view of the tensor-core GEMM's work schedule for an
 * M x N x K product on `sm_count` SMs (CTA pairs = sm_count / 2; 0 means the GB300's
 * 152): the 1xTF32 kernel's for SGEMM_MODE_TF32, the FP16 kernel's for
 * SGEMM_MODE_3XFP16_SCALED, the 3xTF32 kernel's for the other modes (the schedule that
 * applies when solve_ex picks a tensor-core kernel; see sgemm_plan for whether it does).
 * Unit i is written to units[6 i .. 6 i + 5] as: first row of C, first column,
 * columns (rows are always 256, clipped at M), first and one-past-last reduction block
 * (32 elements each, 64 for SGEMM_MODE_3XFP16_SCALED), and the partial-tile slot (-1 when
 * the unit writes C itself; >= 0
 * when it adds into a partial tile that a second kernel sums into C). Units are handed
 * to CTA pairs round-robin in this order. Writes at most `cap` units (units may be NULL
 * with cap 0) and returns the total count, or SGEMM_ERR_ARG.
 */
SGEMM_API int sgemm_plan_units(int M, int N, int K, int mode, int sm_count, int* units,
                               int cap);

/* sgemm_launch_count - number of kernels this library has launched in this process. */
SGEMM_API long long sgemm_launch_count(void);

/*
 * sgemm_set_kernel_events - one-shot timing hook for the calling thread: the next
 * solve/solve_ex call records `start` (a cudaEvent_t) on its stream right before its
 * main kernel (the GEMM, GEMV or GEVM kernel, not the operand split or the final
 * reduction) and `stop` right after it, then forgets both. NULL, NULL clears the hook.
 * Returns SGEMM_OK.
 */
SGEMM_API int sgemm_set_kernel_events(void* start, void* stop);

/*
 * sgemm_selftest_wait_timeout - exercises the kernels' failure path: launches one CTA
 * that waits, with the same bounded wait the GEMM kernels use, on an mbarrier that
 * nothing completes. The wait gives up after limit_ns nanoseconds (1e6 .. 2e9, else
 * SGEMM_ERR_ARG), sets the device error word and returns; this call then waits for the
 * stream and returns what sgemm_device_error reads (SGEMM_ERR_TIMEOUT when the path
 * works) and clears the word. The context stays usable afterwards.
 */
SGEMM_API int sgemm_selftest_wait_timeout(long long limit_ns, void* stream);

/*
 * sgemm_peak_probe - measures a peak arithmetic rate of the current device, for the
 * roofline that the kernels are measured against; the pages have no counterpart (their
 * rooflines quote vendor figures). `probe` is an SGEMM_PROBE_*:
 *   FFMA, FFMA2 - every SM runs 2048 threads of 16 independent register-only FMA chains
 *                 for `iters` steps (scalar fmaf, or packed two-lane FMAs);
 *   TF32_MMA    - every SM pair fills one A and one B^T block in shared memory and issues
 *                 `iters` reduction blocks of four M=256 N=256 K=8 pair MMAs into TMEM,
 *                 the GEMM kernels' instruction form, with nothing else in the way;
 *   F16_MMA     - the same with kind::f16 MMAs on FP16 operands (K=16 per MMA).
 * iters: 1 .. 1048576 for FFMA/FFMA2, 1 .. 262144 for TF32_MMA and F16_MMA, else
 * SGEMM_ERR_ARG.
 * The probe runs on `stream` between two CUDA events; this call waits for the second
 * one, then writes the floating-point operations performed to *flop and the event time
 * to *ms (both required, else SGEMM_ERR_ARG). The device must be idle for a meaningful
 * rate. Returns SGEMM_OK, SGEMM_ERR_TIMEOUT (a bounded wait gave up), SGEMM_ERR_CUDA or
 * SGEMM_ERR_NO_DEVICE.
 */
SGEMM_API int sgemm_peak_probe(int probe, int iters, void* stream, double* flop, float* ms);

/*
 * sgemm_tc_clock_mhz - the SM clock, in MHz, that the last tensor-core launch on the
 * current device ran at (a 3xTF32 or 1xTF32 GEMM, or the TF32_MMA rate probe). CTA 0 of
 * every such launch records its SM's cycle counter (clock64) and the global nanosecond
 * timer when it issues its first MMA and after its last store (the probe: after its MMAs
 * complete); this call reads the record on `stream`, waits for it, and writes the cycles
 * over the nanoseconds, times 1000, to *mhz. It is what the tensor-core rooflines are
 * computed at: the nominal 2070 MHz holds only while the chip has power to spare.
 * Returns SGEMM_OK, SGEMM_ERR_ARG (mhz null), SGEMM_ERR_UNSUPPORTED (no tensor-core
 * launch has completed yet), SGEMM_ERR_CUDA or SGEMM_ERR_NO_DEVICE.
 */
SGEMM_API int sgemm_tc_clock_mhz(void* stream, double* mhz);

/*
 * sgemm_simt_clock_mhz - the same reading for the last CUDA-core launch on the current
 * device (the FFMA GEMM, SGEMM_MODE_FP32_SIMT, or the FFMA/FFMA2 rate probes): thread 0
 * of CTA 0 records its SM's clock64 and the global timer when it starts and when it
 * ends. Arguments and returns as for sgemm_tc_clock_mhz.
 */
SGEMM_API int sgemm_simt_clock_mhz(void* stream, double* mhz);

/*
 * sgemm_release_pool - frees the workspace memory the library's pool holds for the
 * current device beyond what is in use. Waits for the device. Returns SGEMM_OK or
 * SGEMM_ERR_CUDA.
 */
SGEMM_API int sgemm_release_pool(void);

/*
 * solve_row_noalloc - the one-row product C[1 x K] = A[1 x N] . B[N x K] (the M == 1
 * case of solve_ex in SGEMM_MODE_FP32) that allocates no device memory. The pages have
 * no counterpart; it exists for callers that cannot allocate: an application whose own
 * allocator has reserved nearly all device memory up front (a cudaMalloc, or growth of
 * this library's pool, would fail there), one that must account every device byte
 * through its own allocator, or a loop that cannot take an allocation's possible
 * synchronisation.
 *
 * A (N floats), B (N x K, row-major) and C (K floats) are device pointers owned by the
 * caller, as for solve_ex; stream is a cudaStream_t (NULL: legacy default stream).
 * 1 <= N, K <= 8192; larger sizes are rejected with SGEMM_ERR_ARG before anything is
 * enqueued. The split-n partial rows go to a fixed device array of 8 x 8192 floats
 * (256 KiB) that every GPU loading the library holds until the process exits; at most
 * 8 partial rows are used, so when solve_ex would use more, the two may differ in the
 * last bits (both stay within the FP32 contract).
 *
 * The array is part of the library's device code. It is reserved on a device when
 * that code is first loaded there: with CUDA's default lazy module loading, at the
 * first call on that device that needs it (this entry point's first call, or a
 * one-row, one-column or short-reduction product through solve_ex). A caller whose
 * allocator will take nearly all device memory should therefore make one call before
 * that allocator starts. The first successful call on each device looks up the
 * array's device address (with the device current); make that first call before any
 * stream capture. If that set-up fails (SGEMM_ERR_CUDA), nothing is remembered and the
 * next call tries again; the failed call leaves no error in cudaGetLastError(). Every
 * call shares the one array and fully rewrites the part it reads, so no clearing is
 * needed between calls, but calls that overlap on the GPU (different streams, or
 * different threads without ordering) race on it. Returns SGEMM_OK, SGEMM_ERR_ARG,
 * SGEMM_ERR_OVERLAP, SGEMM_ERR_NO_DEVICE or SGEMM_ERR_CUDA. Calls no cudaMalloc,
 * cudaFree or allocating library routine.
 */
SGEMM_API int solve_row_noalloc(const float* A, const float* B, float* C, int N, int K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
