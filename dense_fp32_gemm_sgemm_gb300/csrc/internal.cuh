// Internal interfaces between the C-ABI layer (sgemm_api.cu) and the kernel
// translation units. Nothing here is exported from the shared library.
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

namespace sgemm {

// Per-device facts queried once.
struct DeviceInfo {
    int sm_count = 0;
    int major = 0;
    int minor = 0;
    int smem_optin = 0;  // max dynamic shared memory per block after opt-in, bytes
    int* error_word = nullptr;  // device address of the bounded-wait error word
    bool usable = false;
};

// Records the caller's timing events around the main kernel of one call.
struct KernelTimer {
    cudaEvent_t start = nullptr;
    cudaEvent_t stop = nullptr;
    cudaStream_t stream = nullptr;
    void before() const {
        if (start) cudaEventRecord(start, stream);
    }
    void after() const {
        if (stop) cudaEventRecord(stop, stream);
    }
};

// Raises KERNEL's dynamic shared-memory limit to `bytes` once per device (the attribute
// belongs to the function on each device); later calls return the cached result.
template <auto KERNEL>
cudaError_t set_smem_limit_once(int bytes) {
    constexpr int kDevices = 64;
    static std::once_flag once[kDevices];
    static cudaError_t result[kDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices)
        return cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    std::call_once(once[dev], [bytes, dev] {
        result[dev] = cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    });
    return result[dev];
}

extern std::atomic<long long> g_launches;
inline void count_launch(long long n = 1) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// Values the bounded waits write into the device error word.
enum : int { kErrNone = 0, kErrWaitTimeout = 1 };

// ---- CUDA-core FFMA GEMM (simt_gemm.cu) ----
// Output tile of one CTA; the host uses it for tile counts.
constexpr int kSimtBM = 128;
constexpr int kSimtBN = 128;
// vec: A, B, C 16-byte aligned and N % 4 == 0 and K % 4 == 0.
cudaError_t launch_simt(const float* A, const float* B, float* C, int M, int N, int K, bool vec,
                        cudaStream_t stream, const KernelTimer& timer);

// FFMA on 16 x 64 or 16 x 32 tiles with the reduction split in four inside the CTA (32 x 64
// tiles, unsplit, when rows are not 16-byte aligned), for products too small to fill the
// SMs with 128 x 128 tiles; simt_small_suits tells which.
bool simt_small_suits(int M, int K, int sm_count);
int simt_small_tiles(int M, int K, bool vec, int sm_count);  // its CTA count
cudaError_t launch_simt_small(const float* A, const float* B, float* C, int M, int N, int K,
                              bool vec, int sm_count, cudaStream_t stream,
                              const KernelTimer& timer);

// Register-only FMA rate probe (scalar fmaf, or packed __ffma2_rn) on all SMs, and the
// floating-point operations one launch performs.
cudaError_t launch_ffma_probe(bool packed, int iters, int sm_count, cudaStream_t stream,
                              const KernelTimer& timer);
double ffma_probe_flops(int iters, int sm_count);

// ---- streaming kernels for one-row / one-column / short-reduction shapes (skinny.cu) ----
// N <= kSmallNMax (and M, K > 1): the short-reduction kernel; its CTA count.
constexpr int kSmallNMax = 4;
cudaError_t launch_smalln(const float* A, const float* B, float* C, int M, int N, int K,
                          cudaStream_t stream, const KernelTimer& timer);
int smalln_blocks(int M, int K);
// K == 1: y[m] = sum_n A[m][n] * x[n].
cudaError_t launch_gemv(const float* A, const float* x, float* y, int M, int N, bool vec,
                        cudaStream_t stream, const KernelTimer& timer);
// M == 1: C[k] = sum_n a[n] * B[n][k]. `splits` partial rows go to `partials`
// (splits * K floats) and a second kernel adds them in a fixed order; with splits == 1
// the first kernel writes C directly and `partials` may be null.
int gevm_splits(int N, int K, int sm_count);
cudaError_t launch_gevm(const float* a, const float* B, float* C, int N, int K, bool vec,
                        int splits, float* partials, cudaStream_t stream,
                        const KernelTimer& timer);

// ---- tcgen05 TF32 GEMM (tc_gemm.cu) ----
constexpr int kTcBM = 256;  // output tile of one CTA pair
constexpr int kTcBN = 256;
// Workspace: the rounded operand planes (one plane per operand for 1xTF32, two for
// 3xTF32), the fused split's counters, plus room for the FP32 partial tiles of the
// reduction splits that the schedule on `sm_count` SMs uses, for the whole product or,
// with chunk_rows > 0, for row chunks of at most chunk_rows rows; bytes.
size_t tc_workspace_bytes(int M, int N, int K, int passes, int sm_count, int chunk_rows,
                          bool raw_a);
// With chunk_rows > 0 the partial area holds two sets (for two chunk GEMMs in flight on
// different streams); the floats of one set.
size_t tc_partial_set_floats(int M, int N, int K, int passes, int sm_count, int chunk_rows);
// The GEMM's unit list (6 ints per unit, see sgemm_plan_units); returns the unit count.
int tc_schedule_units(int M, int N, int K, int passes, int sm_count, int* out, int cap);
// Where the planes and the partial area sit in a workspace.
struct TcLayout {
    int lda, ldbt;  // row pitches (floats) of the A and B^T planes
    float *a_hi, *a_lo, *b_hi, *b_lo, *partials;
    int* counters;  // progress counters of a GEMM that splits A itself
    // 3xTF32 with a TMA-legal A (16-byte aligned, N % 4 == 0): A itself, used as the hi
    // plane (the tensor core truncates it); the layout then has no a_hi plane (null)
    const float* a_raw = nullptr;
};
// a_raw: tc_raw_hi of the A that will be multiplied (the workspace must have been sized
// with raw_a = (a_raw != null)).
TcLayout tc_layout(float* workspace, int M, int N, int K, int passes, const float* a_raw);
// A when the 3xTF32 GEMM can load it as its own hi plane, else null (for TcLayout::a_raw).
const float* tc_raw_hi(const float* A, int N, int passes);
// Operand pre-pass: rounds (1xTF32) or splits (3xTF32) the M rows of A into rows
// [a_row0, a_row0 + M) of the A planes (only lo when L.a_raw is set), and/or B (N x K)
// into the B^T planes. A or B may be null to skip that operand. One launch.
// With A_first (the whole A, for a GEMM that splits A itself) and B, the launch also
// prepares the first 1024-column chunk of A's first first_rows rows and marks it done in
// the counters.
cudaError_t tc_prep(const float* A, int M, int a_row0, const float* B, int N, int K, int passes,
                    const TcLayout& L, int sm_count, cudaStream_t stream,
                    const float* A_first = nullptr, int first_rows = 0);
// GEMM of rows [row0, row0 + rows) of the A planes against the B^T planes into C_rows
// (rows x K, row-major), plus the split reduction when the schedule splits tiles. With
// A_fused (those rows of A; N % 4 == 0 and 16-byte aligned, else cudaErrorInvalidValue)
// the GEMM kernel splits (3xTF32) or rounds (1xTF32) A into the planes itself.
cudaError_t tc_gemm_rows(const TcLayout& L, int row0, int rows, int N, int K, int passes,
                         float* C_rows, int sm_count, cudaStream_t stream,
                         const KernelTimer& timer, int* err, const float* A_fused = nullptr);
// The whole product: pre-pass then GEMM.
cudaError_t launch_tc(const float* A, const float* B, float* C, int M, int N, int K, int passes,
                      float* workspace, int sm_count, cudaStream_t stream,
                      const KernelTimer& timer, int* err);

// Shared-memory-resident pair MMA rate probe (tcgen05 kind::tf32, or kind::f16 with FP16
// operands; M=256 N=256) on every SM pair, and the floating-point operations one launch
// performs.
cudaError_t launch_mma_probe(bool f16, int iters, int sm_count, int* err, cudaStream_t stream,
                             const KernelTimer& timer);
double mma_probe_flops(bool f16, int iters, int sm_count);

// The FP16 three-product path (SGEMM_MODE_3XFP16_SCALED): workspace bytes, the launch
// (pre-passes, GEMM, split reduction) and its schedule (as tc_schedule_units).
size_t tc16_workspace_bytes(int M, int N, int K, int sm_count);
cudaError_t launch_tc16(const float* A, const float* B, float* C, int M, int N, int K,
                        void* workspace, int sm_count, cudaStream_t stream,
                        const KernelTimer& timer, int* err);
int tc16_schedule_units(int M, int N, int K, int sm_count, int* out, int cap);

// The clock record of the last tensor-core GEMM or TF32 probe launch on this device:
// CTA 0's globaltimer ns and clock64 cycles at its first MMA ([0], [1]) and after its
// last store ([2], [3]); all zero before the first launch. Synchronises `stream`.
cudaError_t tc_clock_record(cudaStream_t stream, unsigned long long (&out)[4]);
// The same for the last CUDA-core GEMM or FFMA probe launch (thread 0 of CTA 0, from its
// start to its end).
cudaError_t simt_clock_record(cudaStream_t stream, unsigned long long (&out)[4]);

// One CTA whose bounded wait on a never-completed mbarrier gives up after limit_ns
// and sets *err (the device error word).
cudaError_t launch_wait_selftest(long long limit_ns, int* err, cudaStream_t stream);

}  // namespace sgemm
