// Streaming kernels for the one-row and one-column shapes. With M == 1 or K == 1 the
// product does 2 flops per element of the large operand, so the time is the time to
// read that operand once from HBM; these kernels are built to do exactly that.
//
//  * GEMV (K == 1): y[m] = sum_n A[m][n] * x[n]. A CTA streams 2 consecutive rows of A
//    (one contiguous block) with every thread holding sixteen 128-bit loads in flight
//    and x in registers, then adds each row's partial sums in a fixed order.
//  * GEVM (M == 1): C[k] = sum_n a[n] * B[n][k]. Each CTA owns a 64-column strip of B
//    and one slice of the n range; its threads stream rows of the strip (128-bit loads
//    along k), and the row groups are added in shared memory in a fixed order. When
//    the strips alone cannot fill the GPU, the n range is split across CTAs and a
//    second kernel adds the partial rows in split order. No float atomics anywhere, so
//    results are bitwise reproducible run to run.
//  * Short reductions (N <= kSmallNMax = 4, M, K > 1): C has M x K elements but each
//    takes only N fused multiply-adds, so writing C once is the cost (from N = 6 up the
//    tensor-core path is faster on 8192 x N x 8192). Each CTA owns a
//    64-row x 128-column block of C: it stages that block's rows of A and its N x 128
//    slice of B in shared memory, then each warp computes its 8 rows one at a time,
//    lane l owning columns c0 + l + 32 j, and writes 32 consecutive floats per store
//    instruction, at any alignment. Every C[m][k] is one FP32 accumulator updated by fmaf with n
//    ascending, the arithmetic of the CUDA-core GEMM.
#include <atomic>
#include <mutex>

#include "internal.cuh"
#include "sgemm.h"

namespace sgemm {
namespace {

constexpr int GEMV_THREADS = 256;
constexpr int GEMV_ROWS = 2;  // rows of A per CTA
constexpr int GEVM_THREADS = 256;
constexpr int GEVM_COLS = 64;

__device__ __forceinline__ float4 ld_stream4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

// K == 1: a CTA of 256 threads reads GEMV_ROWS consecutive rows of A (one contiguous
// block of memory). Thread t covers columns t + 256 j (float4 columns when VEC) and holds
// its values of x in registers; it issues all its loads of the block's rows before using
// them (16 x 128-bit or 2 x 32 x 32-bit in flight), sums its share of a row in n order,
// and a row's partial sums are combined by a fixed butterfly within each warp and in
// warp order across warps. (Swept on GB300 with non-zero data: one row at a time reads
// at 5.0 TB/s, two rows in flight at 6.2 TB/s.)
template <bool VEC>
__global__ void __launch_bounds__(GEMV_THREADS)
    gemv_kernel(const float* __restrict__ A, const float* __restrict__ x, float* __restrict__ y,
                int M, int N) {
    constexpr int J = VEC ? 8192 / (GEMV_THREADS * 4) : 8192 / GEMV_THREADS;
    __shared__ float red[GEMV_THREADS / 32][GEMV_ROWS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * GEMV_ROWS;
    float s[GEMV_ROWS];
    if constexpr (VEC) {
        const int n4 = N >> 2;
        const float4* x4 = reinterpret_cast<const float4*>(x);
        float4 xv[J];
#pragma unroll
        for (int j = 0; j < J; ++j)
            xv[j] = tid + GEMV_THREADS * j < n4 ? __ldg(x4 + tid + GEMV_THREADS * j)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 av[GEMV_ROWS][J];
#pragma unroll
        for (int u = 0; u < GEMV_ROWS; ++u) {
            const float4* a = reinterpret_cast<const float4*>(A + size_t(r0 + u) * N);
#pragma unroll
            for (int j = 0; j < J; ++j)
                av[u][j] = r0 + u < M && tid + GEMV_THREADS * j < n4
                               ? __ldcs(a + tid + GEMV_THREADS * j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < GEMV_ROWS; ++u) {
            s[u] = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                s[u] = fmaf(av[u][j].x, xv[j].x, s[u]);
                s[u] = fmaf(av[u][j].y, xv[j].y, s[u]);
                s[u] = fmaf(av[u][j].z, xv[j].z, s[u]);
                s[u] = fmaf(av[u][j].w, xv[j].w, s[u]);
            }
        }
    } else {
        float xv[J];
#pragma unroll
        for (int j = 0; j < J; ++j)
            xv[j] = tid + GEMV_THREADS * j < N ? __ldg(x + tid + GEMV_THREADS * j) : 0.f;
#pragma unroll
        for (int u = 0; u < GEMV_ROWS; ++u) {
            const float* a = A + size_t(r0 + u) * N;
            float av[J];
#pragma unroll
            for (int j = 0; j < J; ++j)
                av[j] = r0 + u < M && tid + GEMV_THREADS * j < N ? __ldcs(a + tid + GEMV_THREADS * j)
                                                                 : 0.f;
            s[u] = 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) s[u] = fmaf(av[j], xv[j], s[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < GEMV_ROWS; ++u) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s[u] += __shfl_xor_sync(0xffffffffu, s[u], o);
        if (lane == 0) red[warp][u] = s[u];
    }
    __syncthreads();
    if (tid < GEMV_ROWS && r0 + tid < M) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < GEMV_THREADS / 32; ++w) t += red[w][tid];
        y[r0 + tid] = t;
    }
}

// One CTA: columns [blockIdx.x * 64, +64) of B, rows [split * rows_per_split, +rows).
template <bool VEC>
__global__ void __launch_bounds__(GEVM_THREADS)
    gevm_kernel(const float* __restrict__ a, const float* __restrict__ B, float* __restrict__ out,
                int N, int K, int rows_per_split) {
    constexpr int LANES = VEC ? GEVM_COLS / 4 : GEVM_COLS;
    constexpr int GROUPS = GEVM_THREADS / LANES;
    __shared__ float red[GROUPS][GEVM_COLS];
    const int lane = threadIdx.x % LANES, g = threadIdx.x / LANES;
    const int split = blockIdx.y;
    const int n_begin = split * rows_per_split;
    const int n_end = min(N, n_begin + rows_per_split);
    const int col_base = blockIdx.x * GEVM_COLS;
    if constexpr (VEC) {
        const int col = col_base + lane * 4;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < K) {
#pragma unroll 4
            for (int n = n_begin + g; n < n_end; n += GROUPS) {
                const float av = __ldg(a + n);
                const float4 b = ld_stream4(B + (size_t)n * K + col);
                s.x = fmaf(av, b.x, s.x);
                s.y = fmaf(av, b.y, s.y);
                s.z = fmaf(av, b.z, s.z);
                s.w = fmaf(av, b.w, s.w);
            }
        }
        red[g][lane * 4 + 0] = s.x;
        red[g][lane * 4 + 1] = s.y;
        red[g][lane * 4 + 2] = s.z;
        red[g][lane * 4 + 3] = s.w;
    } else {
        const int col = col_base + lane;
        float s = 0.f;
        if (col < K) {
#pragma unroll 4
            for (int n = n_begin + g; n < n_end; n += GROUPS)
                s = fmaf(__ldg(a + n), __ldcs(B + (size_t)n * K + col), s);
        }
        red[g][lane] = s;
    }
    __syncthreads();
    if (threadIdx.x < GEVM_COLS) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < GROUPS; ++r) s += red[r][threadIdx.x];
        const int col = col_base + threadIdx.x;
        if (col < K) out[(size_t)split * K + col] = s;
    }
}

__global__ void gevm_reduce_kernel(const float* __restrict__ partials, float* __restrict__ C,
                                   int K, int splits) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= K) return;
    float s = 0.f;
    for (int i = 0; i < splits; ++i) s += partials[(size_t)i * K + k];
    C[k] = s;
}

constexpr int SMALLN_ROWS = 64;   // rows of C per CTA (8 per warp)
constexpr int SMALLN_COLS = 128;  // columns of C per CTA (4 per lane, 32 apart)

__global__ void __launch_bounds__(256, 8)
    smalln_kernel(const float* __restrict__ A, const float* __restrict__ B,
                  float* __restrict__ C, int M, int N, int K) {
    // the CTA's rows of A (contiguous in memory: rows x N floats) and its N x 128 slice of
    // B, staged once; then every warp computes and stores 8 rows of the block
    __shared__ float As[SMALLN_ROWS * kSmallNMax];
    __shared__ float Bs[kSmallNMax * SMALLN_COLS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col0 = blockIdx.x * SMALLN_COLS;
    const int row0 = blockIdx.y * SMALLN_ROWS;
    const int rows = M - row0 < SMALLN_ROWS ? M - row0 : SMALLN_ROWS;
    const float* a_src = A + size_t(row0) * N;
    for (int i = tid; i < rows * N; i += blockDim.x) As[i] = __ldg(a_src + i);
    for (int i = tid; i < N * SMALLN_COLS; i += blockDim.x) {
        const int n = i / SMALLN_COLS, c = i % SMALLN_COLS;
        Bs[i] = col0 + c < K ? __ldg(B + size_t(n) * K + col0 + c) : 0.0f;
    }
    __syncthreads();
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
        const int r = warp * 8 + i;
        if (r >= rows) break;  // warp-uniform
        const float* ar = As + r * N;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
        for (int n = 0; n < N; ++n) {
            const float av = ar[n];
            const float* bn = Bs + n * SMALLN_COLS + lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(av, bn[32 * j], acc[j]);
        }
        float* crow = C + size_t(row0 + r) * K + col0 + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (col0 + lane + 32 * j < K) __stcs(crow + 32 * j, acc[j]);
    }
}

}  // namespace

cudaError_t launch_smalln(const float* A, const float* B, float* C, int M, int N, int K,
                          cudaStream_t stream, const KernelTimer& timer) {
    const dim3 grid((K + SMALLN_COLS - 1) / SMALLN_COLS, (M + SMALLN_ROWS - 1) / SMALLN_ROWS);
    timer.before();
    smalln_kernel<<<grid, 256, 0, stream>>>(A, B, C, M, N, K);
    cudaError_t err = cudaGetLastError();
    timer.after();
    count_launch();
    return err;
}

int smalln_blocks(int M, int K) {
    return ((K + SMALLN_COLS - 1) / SMALLN_COLS) * ((M + SMALLN_ROWS - 1) / SMALLN_ROWS);
}

cudaError_t launch_gemv(const float* A, const float* x, float* y, int M, int N, bool vec,
                        cudaStream_t stream, const KernelTimer& timer) {
    const int blocks = (M + GEMV_ROWS - 1) / GEMV_ROWS;
    timer.before();
    if (vec)
        gemv_kernel<true><<<blocks, GEMV_THREADS, 0, stream>>>(A, x, y, M, N);
    else
        gemv_kernel<false><<<blocks, GEMV_THREADS, 0, stream>>>(A, x, y, M, N);
    cudaError_t err = cudaGetLastError();
    timer.after();
    count_launch();
    return err;
}

int gevm_splits(int N, int K, int sm_count) {
    const int strips = (K + GEVM_COLS - 1) / GEVM_COLS;
    // about six 256-thread CTAs per SM keep enough 128-bit loads in flight
    const int target = 6 * (sm_count > 0 ? sm_count : 1);
    if (strips >= target) return 1;
    int splits = (target + strips - 1) / strips;
    const int max_by_rows = N / 64;  // keep at least 64 rows of B per CTA
    if (splits > max_by_rows) splits = max_by_rows;
    if (splits > 64) splits = 64;
    return splits < 1 ? 1 : splits;
}

cudaError_t launch_gevm(const float* a, const float* B, float* C, int N, int K, bool vec,
                        int splits, float* partials, cudaStream_t stream,
                        const KernelTimer& timer) {
    const int strips = (K + GEVM_COLS - 1) / GEVM_COLS;
    const int rows_per_split = (N + splits - 1) / splits;
    float* out = splits == 1 ? C : partials;
    const dim3 grid(strips, splits);
    timer.before();
    if (vec)
        gevm_kernel<true><<<grid, GEVM_THREADS, 0, stream>>>(a, B, out, N, K, rows_per_split);
    else
        gevm_kernel<false><<<grid, GEVM_THREADS, 0, stream>>>(a, B, out, N, K, rows_per_split);
    cudaError_t err = cudaGetLastError();
    timer.after();
    count_launch();
    if (err != cudaSuccess || splits == 1) return err;
    gevm_reduce_kernel<<<(K + 255) / 256, 256, 0, stream>>>(partials, C, K, splits);
    count_launch();
    return cudaGetLastError();
}

}  // namespace sgemm

// ------------------------------------------------------------------------------------
// Allocation-free one-row product (solve_row_noalloc).
//
// Some callers cannot allocate device memory at all: an application whose allocator
// has reserved nearly all of HBM up front (so any cudaMalloc, or growth of this
// library's pool, would fail), one that must account every device byte through its
// own allocator, or a latency-critical loop that cannot take an allocation's possible
// synchronisation. For them the split-n partial rows of the one-row product live in a
// fixed array in the library's device image instead of the pool.
namespace sgemm {
namespace {

constexpr int kNoAllocMaxDim = 8192;
constexpr int kNoAllocMaxSplits = 8;
// 8 partial rows of the widest allowed K: 65,536 floats (256 KiB) per device.
constexpr int kNoAllocScratchFloats = kNoAllocMaxSplits * kNoAllocMaxDim;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_partials[kNoAllocScratchFloats];

struct NoAllocDevice {
    float* partials = nullptr;  // device address of g_noalloc_partials on this device
    int sm_count = 0;
    std::atomic<bool> ready{false};  // set only after a successful set-up
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex[kNoAllocMaxDevices];

// Set-up of one device, with that device current: the array's name is only a host-side
// stand-in, so the device address has to be looked up before a kernel can be given it.
// With CUDA's lazy module loading the lookup is also what loads this file's device code,
// and with it the array, onto the device. A failure is not remembered: the error is
// cleared from the runtime's last-error state and the next call tries again (the load
// can fail while another allocator holds nearly all device memory, and succeed once it
// has given some back). Returns SGEMM_OK, SGEMM_ERR_NO_DEVICE or SGEMM_ERR_CUDA.
int noalloc_setup(int dev) {
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (d.ready.load(std::memory_order_acquire)) return SGEMM_OK;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex[dev]);
    if (d.ready.load(std::memory_order_relaxed)) return SGEMM_OK;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return SGEMM_ERR_NO_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return SGEMM_ERR_CUDA;
    }
    d.partials = static_cast<float*>(p);
    d.sm_count = sms;
    d.ready.store(true, std::memory_order_release);
    return SGEMM_OK;
}

bool noalloc_overlap(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

}  // namespace
}  // namespace sgemm

extern "C" int solve_row_noalloc(const float* A, const float* B, float* C, int N, int K,
                                 void* stream) {
    using namespace sgemm;
    if (N < 1 || K < 1 || N > kNoAllocMaxDim || K > kNoAllocMaxDim) return SGEMM_ERR_ARG;
    if (!A || !B || !C) return SGEMM_ERR_ARG;
    if (noalloc_overlap(C, size_t(K) * sizeof(float), A, size_t(N) * sizeof(float)) ||
        noalloc_overlap(C, size_t(K) * sizeof(float), B, size_t(N) * K * sizeof(float)))
        return SGEMM_ERR_OVERLAP;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return SGEMM_ERR_NO_DEVICE;
    }
    const int setup = noalloc_setup(dev);
    if (setup != SGEMM_OK) return setup;
    const NoAllocDevice& d = g_noalloc_dev[dev];
    int splits = gevm_splits(N, K, d.sm_count);
    if (splits > kNoAllocMaxSplits) splits = kNoAllocMaxSplits;
    if (size_t(splits) * K > size_t(kNoAllocScratchFloats)) return SGEMM_ERR_ARG;  // cannot happen for K <= 8192
    // same loader choice as solve_ex, so both sum in the same order when the split
    // counts agree. (The GEVM kernel writes C with 4-byte stores whatever the loader; C's
    // alignment is in the condition only because solve_ex's "aligned" flag includes it,
    // so that both entry points pick the same loader for the same pointers.)
    const bool vec = (reinterpret_cast<uintptr_t>(A) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(B) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && K % 4 == 0;
    const KernelTimer no_timer;
    const cudaError_t err = launch_gevm(A, B, C, N, K, vec, splits, d.partials,
                                        static_cast<cudaStream_t>(stream), no_timer);
    return err == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

