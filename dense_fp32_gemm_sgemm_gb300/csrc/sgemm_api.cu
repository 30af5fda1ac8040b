// The C ABI declared in include/sgemm.h: argument checks, kernel selection, the
// workspace pool, per-thread stream/status state and the query calls.
//
// The entry point keeps the signature of "LeetGPU | 02_Matrix_Multiplication",
// section "Implementation Requirements" (solve with device pointers, result in C);
// everything else here is this library's own.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.cuh"
#include "sgemm.h"

namespace sgemm {

std::atomic<long long> g_launches{0};

namespace {

constexpr int kMaxDim = 8192;
constexpr int kMaxDevices = 64;
// FP32 mode runs on the CUDA cores up to kSimtTinyWork multiply-adds, and up to
// kSimtMaxWork when the reduction is at most kSimtMaxReduction long
constexpr int64_t kSimtTinyWork = int64_t(1) << 22;
constexpr int64_t kSimtMaxWork = int64_t(1) << 27;
constexpr int kSimtMaxReduction = 1024;

__device__ int g_error_word;

thread_local cudaStream_t tl_stream = nullptr;
thread_local int tl_status = SGEMM_OK;
thread_local cudaEvent_t tl_ev_start = nullptr;
thread_local cudaEvent_t tl_ev_stop = nullptr;

DeviceInfo g_info[kMaxDevices];
std::once_flag g_info_once[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];
std::once_flag g_pool_once[kMaxDevices];

void init_device(int dev) {
    DeviceInfo& d = g_info[dev];
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
        d.usable = false;
        return;
    }
    // The kernels are built for sm_103a only.
    if (d.major != 10 || d.minor != 3) {
        d.usable = false;
        return;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
        d.usable = false;
        return;
    }
    d.error_word = static_cast<int*>(p);
    d.usable = true;
}

const DeviceInfo* current_device(int* dev_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::call_once(g_info_once[dev], init_device, dev);
    if (!g_info[dev].usable) return nullptr;
    if (dev_out) *dev_out = dev;
    return &g_info[dev];
}

cudaError_t pool_for(int dev, cudaMemPool_t* out) {
    static cudaError_t pool_err[kMaxDevices];
    std::call_once(g_pool_once[dev], [dev] {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        pool_err[dev] = cudaMemPoolCreate(&g_pool[dev], &props);
        if (pool_err[dev] == cudaSuccess) {
            // Keep freed blocks for reuse instead of returning them at every sync.
            uint64_t keep = UINT64_MAX;
            pool_err[dev] =
                cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
        }
    });
    *out = g_pool[dev];
    return pool_err[dev];
}

// Stream-ordered scratch from the library pool, released on the same stream.
struct Scratch {
    void* ptr = nullptr;
    cudaStream_t stream = nullptr;
    cudaError_t alloc(int dev, size_t bytes, cudaStream_t s) {
        cudaMemPool_t pool;
        cudaError_t err = pool_for(dev, &pool);
        if (err != cudaSuccess) return err;
        stream = s;
        return cudaMallocFromPoolAsync(&ptr, bytes, pool, s);
    }
    ~Scratch() {
        if (ptr) cudaFreeAsync(ptr, stream);
    }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

int check_args(const float* A, const float* B, const float* C, int M, int N, int K, int mode) {
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_ARG;
    if (!A || !B || !C) return SGEMM_ERR_ARG;
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_3XFP16_SCALED) return SGEMM_ERR_ARG;
    const size_t a_bytes = size_t(M) * N * sizeof(float);
    const size_t b_bytes = size_t(N) * K * sizeof(float);
    const size_t c_bytes = size_t(M) * K * sizeof(float);
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, B, b_bytes))
        return SGEMM_ERR_OVERLAP;
    return SGEMM_OK;
}

// Kernel choice for a shape. Host-only; shared by sgemm_plan and solve_ex.
int choose_kernel(int M, int N, int K, int mode, bool /*aligned*/) {
    switch (mode) {
        case SGEMM_MODE_FP32_SIMT:
            return SGEMM_KERNEL_SIMT;
        case SGEMM_MODE_FP32_3XTF32:
            return SGEMM_KERNEL_TC_3XTF32;
        case SGEMM_MODE_3XFP16_SCALED:
            return SGEMM_KERNEL_TC_3XFP16;
        default:
            break;
    }
    // one-row / one-column shapes stream their big operand, and short reductions write
    // C at HBM speed, in every mode: FP32 FMA is as fast as TF32 there, and meets the
    // FP32 contract
    if (M == 1 && K > 1) return SGEMM_KERNEL_GEVM;
    if (K == 1) return SGEMM_KERNEL_GEMV;
    if (N <= kSmallNMax) return SGEMM_KERNEL_SMALLN;
    if (mode == SGEMM_MODE_TF32) return SGEMM_KERNEL_TC_1XTF32;
    // FP32-accurate: small products run on the CUDA cores in one launch; the segmented
    // 3xTF32 kernel (pre-pass, GEMM and, for few tiles, a split reduction) is faster from
    // about 2^27 multiply-adds up (measured: 512^3 12.4 against 18.9 us, 640^3 22.6
    // against 22.3 us), and for long reductions over few output tiles, which the CUDA-core
    // kernel does not split.
    const int64_t work = int64_t(M) * N * K;
    if (work <= kSimtTinyWork || (work <= kSimtMaxWork && N <= kSimtMaxReduction))
        return SGEMM_KERNEL_SIMT;
    return SGEMM_KERNEL_TC_3XTF32;
}

// Output tiles of the kernel for this shape (for the FFMA kernel on a GB300's 152 SMs;
// vec: its 16-byte copy path).
int tiles_for(int kernel, int M, int K, bool vec) {
    switch (kernel) {
        case SGEMM_KERNEL_SIMT:
            if (simt_small_suits(M, K, 152)) return simt_small_tiles(M, K, vec, 152);
            return ((M + kSimtBM - 1) / kSimtBM) * ((K + kSimtBN - 1) / kSimtBN);
        case SGEMM_KERNEL_GEMV:
            return M;
        case SGEMM_KERNEL_GEVM:
            return (K + 63) / 64;
        case SGEMM_KERNEL_SMALLN:
            return smalln_blocks(M, K);
        case SGEMM_KERNEL_TC_1XTF32:
        case SGEMM_KERNEL_TC_3XTF32:
        case SGEMM_KERNEL_TC_3XFP16:
            return ((M + kTcBM - 1) / kTcBM) * ((K + kTcBN - 1) / kTcBN);
        default:
            return 0;
    }
}

KernelTimer take_timer(cudaStream_t stream) {
    KernelTimer t;
    t.start = tl_ev_start;
    t.stop = tl_ev_stop;
    t.stream = stream;
    tl_ev_start = nullptr;
    tl_ev_stop = nullptr;
    return t;
}

int run(const float* A, const float* B, float* C, int M, int N, int K, int mode,
        cudaStream_t stream) {
    int rc = check_args(A, B, C, M, N, K, mode);
    if (rc != SGEMM_OK) return rc;
    int dev = -1;
    const DeviceInfo* info = current_device(&dev);
    if (!info) return SGEMM_ERR_NO_DEVICE;
    const bool aligned = aligned16(A) && aligned16(B) && aligned16(C);
    const int kernel = choose_kernel(M, N, K, mode, aligned);
    if (kernel < 0) return kernel;
    const KernelTimer timer = take_timer(stream);
    cudaError_t err = cudaSuccess;
    switch (kernel) {
        case SGEMM_KERNEL_SIMT:
            if (simt_small_suits(M, K, info->sm_count))
                err = launch_simt_small(A, B, C, M, N, K, aligned && N % 4 == 0 && K % 4 == 0,
                                        info->sm_count, stream, timer);
            else
                err = launch_simt(A, B, C, M, N, K, aligned && N % 4 == 0 && K % 4 == 0, stream,
                                  timer);
            break;
        case SGEMM_KERNEL_GEMV:
            // B is the N-vector x, C the M-vector y.
            err = launch_gemv(A, B, C, M, N, aligned && N % 4 == 0, stream, timer);
            break;
        case SGEMM_KERNEL_SMALLN:
            err = launch_smalln(A, B, C, M, N, K, stream, timer);
            break;
        case SGEMM_KERNEL_GEVM: {
            // A is the N-vector a.
            const int splits = gevm_splits(N, K, info->sm_count);
            Scratch partials;
            if (splits > 1) {
                err = partials.alloc(dev, size_t(splits) * K * sizeof(float), stream);
                if (err != cudaSuccess) break;
            }
            err = launch_gevm(A, B, C, N, K, aligned && K % 4 == 0, splits,
                              static_cast<float*>(partials.ptr), stream, timer);
            break;
        }
        case SGEMM_KERNEL_TC_1XTF32:
        case SGEMM_KERNEL_TC_3XTF32: {
            const int passes = kernel == SGEMM_KERNEL_TC_3XTF32 ? 3 : 1;
            Scratch ws;
            err = ws.alloc(dev,
                           tc_workspace_bytes(M, N, K, passes, info->sm_count, 0,
                                              tc_raw_hi(A, N, passes) != nullptr),
                           stream);
            if (err != cudaSuccess) break;
            err = launch_tc(A, B, C, M, N, K, passes, static_cast<float*>(ws.ptr), info->sm_count,
                            stream, timer, info->error_word);
            break;
        }
        case SGEMM_KERNEL_TC_3XFP16: {
            Scratch ws;
            err = ws.alloc(dev, tc16_workspace_bytes(M, N, K, info->sm_count), stream);
            if (err != cudaSuccess) break;
            err = launch_tc16(A, B, C, M, N, K, ws.ptr, info->sm_count, stream, timer,
                              info->error_word);
            break;
        }
        default:
            return SGEMM_ERR_UNSUPPORTED;
    }
    return err == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

// Per-device streams for the host round trip: uploads, downloads, operand splits, and a
// second compute stream beside the caller's.
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr, prep = nullptr, comp = nullptr;
    cudaError_t status = cudaErrorNotReady;
};
CopyStreams g_copy[kMaxDevices];
std::once_flag g_copy_once[kMaxDevices];

const CopyStreams& copy_streams(int dev) {
    std::call_once(g_copy_once[dev], [dev] {
        CopyStreams& c = g_copy[dev];
        c.status = cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking);
        if (c.status == cudaSuccess) c.status = cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking);
        if (c.status == cudaSuccess) c.status = cudaStreamCreateWithFlags(&c.prep, cudaStreamNonBlocking);
        if (c.status == cudaSuccess) c.status = cudaStreamCreateWithFlags(&c.comp, cudaStreamNonBlocking);
    });
    return g_copy[dev];
}

// The host round trip for the tensor-core kernels, pipelined over row chunks of A and
// C: B is uploaded first, then A in chunks of kChunkRows rows (copy stream `in`); each
// operand is split on stream `prep` as soon as it has arrived, each chunk's GEMM runs on
// the caller's stream or stream `comp`, alternately, once its rows are split, and each
// chunk of C goes back on copy stream `out` once computed; events order the five
// streams. A chunk's split runs beside the previous chunk's GEMM, and consecutive chunk
// GEMMs overlap, on the SMs a chunk's last round leaves idle (at K = 4096 a 1024-row
// chunk is 64 pair tiles: one round with 12 of 76 pairs free). Each of the two compute
// streams has its own set of split-reduction partials. Waits for everything before it
// returns.
int solve_host_pipelined(const float* hA, const float* hB, float* hC, int M, int N, int K,
                         int passes, int dev, const DeviceInfo* info, cudaStream_t s) {
    constexpr int kChunkRows = 1024;
    constexpr int kChunks = (kMaxDim + kChunkRows - 1) / kChunkRows;
    const CopyStreams& cs = copy_streams(dev);
    if (cs.status != cudaSuccess) return SGEMM_ERR_CUDA;
    const int chunk_rows = kChunkRows;
    const int nc = (M + chunk_rows - 1) / chunk_rows;
    const size_t a_bytes = size_t(M) * N * sizeof(float);
    const size_t b_bytes = size_t(N) * K * sizeof(float);
    const size_t c_bytes = size_t(M) * K * sizeof(float);
    cudaEvent_t ev_ready = nullptr, ev_b = nullptr, ev_done = nullptr, ev_comp = nullptr;
    cudaEvent_t ev_a[kChunks] = {}, ev_p[kChunks] = {}, ev_c[kChunks] = {};
    bool ok = cudaEventCreateWithFlags(&ev_ready, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_b, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_done, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&ev_comp, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < nc; ++c)
        ok = cudaEventCreateWithFlags(&ev_a[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&ev_p[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&ev_c[c], cudaEventDisableTiming) == cudaSuccess;
    int rc = ok ? SGEMM_OK : SGEMM_ERR_CUDA;
    {
        Scratch dA, dB, dC, ws;
        if (rc == SGEMM_OK &&
            (dA.alloc(dev, a_bytes, s) != cudaSuccess || dB.alloc(dev, b_bytes, s) != cudaSuccess ||
             dC.alloc(dev, c_bytes, s) != cudaSuccess ||
             ws.alloc(dev,
                      tc_workspace_bytes(M, N, K, passes, info->sm_count, chunk_rows,
                                         tc_raw_hi(static_cast<const float*>(dA.ptr), N, passes) !=
                                             nullptr),
                      s) !=
                 cudaSuccess))
            rc = SGEMM_ERR_CUDA;
        if (rc == SGEMM_OK) {
            const float* A = static_cast<const float*>(dA.ptr);
            const float* B = static_cast<const float*>(dB.ptr);
            float* C = static_cast<float*>(dC.ptr);
            const TcLayout L =
                tc_layout(static_cast<float*>(ws.ptr), M, N, K, passes, tc_raw_hi(A, N, passes));
            const size_t part_set =
                tc_partial_set_floats(M, N, K, passes, info->sm_count, chunk_rows);
            const KernelTimer timer = take_timer(s);
            cudaError_t e = cudaEventRecord(ev_ready, s);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, ev_ready, 0);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_ready, 0);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.prep, ev_ready, 0);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.comp, ev_ready, 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(dB.ptr, hB, b_bytes, cudaMemcpyHostToDevice, cs.in);
            if (e == cudaSuccess) e = cudaEventRecord(ev_b, cs.in);
            for (int c = 0; e == cudaSuccess && c < nc; ++c) {
                const int r0 = c * chunk_rows, rows = M - r0 < chunk_rows ? M - r0 : chunk_rows;
                e = cudaMemcpyAsync(static_cast<float*>(dA.ptr) + size_t(r0) * N, hA + size_t(r0) * N,
                                    size_t(rows) * N * sizeof(float), cudaMemcpyHostToDevice, cs.in);
                if (e == cudaSuccess) e = cudaEventRecord(ev_a[c], cs.in);
            }
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.prep, ev_b, 0);
            if (e == cudaSuccess)
                e = tc_prep(nullptr, 0, 0, B, N, K, passes, L, info->sm_count, cs.prep);
            for (int c = 0; e == cudaSuccess && c < nc; ++c) {
                const int r0 = c * chunk_rows, rows = M - r0 < chunk_rows ? M - r0 : chunk_rows;
                e = cudaStreamWaitEvent(cs.prep, ev_a[c], 0);
                if (e == cudaSuccess)
                    e = tc_prep(A + size_t(r0) * N, rows, r0, nullptr, N, K, passes, L,
                                info->sm_count, cs.prep);
                if (e == cudaSuccess) e = cudaEventRecord(ev_p[c], cs.prep);
            }
            for (int c = 0; e == cudaSuccess && c < nc; ++c) {
                const int r0 = c * chunk_rows, rows = M - r0 < chunk_rows ? M - r0 : chunk_rows;
                cudaStream_t cs_c = (c & 1) ? cs.comp : s;
                TcLayout Lc = L;
                Lc.partials = L.partials + (c & 1) * part_set;
                e = cudaStreamWaitEvent(cs_c, ev_p[c], 0);
                if (e == cudaSuccess)
                    e = tc_gemm_rows(Lc, r0, rows, N, K, passes, C + size_t(r0) * K,
                                     info->sm_count, cs_c, c == 0 ? timer : KernelTimer{},
                                     info->error_word);
                if (e == cudaSuccess) e = cudaEventRecord(ev_c[c], cs_c);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_c[c], 0);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(hC + size_t(r0) * K, C + size_t(r0) * K,
                                        size_t(rows) * K * sizeof(float), cudaMemcpyDeviceToHost,
                                        cs.out);
            }
            if (e == cudaSuccess) e = cudaEventRecord(ev_comp, cs.comp);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_comp, 0);
            if (e == cudaSuccess) e = cudaEventRecord(ev_done, cs.out);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_done, 0);
            if (e != cudaSuccess) rc = SGEMM_ERR_CUDA;
        }
        // nothing may still use the buffers when the pool takes them back
        if (cudaStreamSynchronize(cs.in) != cudaSuccess) rc = SGEMM_ERR_CUDA;
        if (cudaStreamSynchronize(cs.out) != cudaSuccess) rc = SGEMM_ERR_CUDA;
        if (cudaStreamSynchronize(cs.prep) != cudaSuccess) rc = SGEMM_ERR_CUDA;
        if (cudaStreamSynchronize(cs.comp) != cudaSuccess) rc = SGEMM_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) rc = SGEMM_ERR_CUDA;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess && rc == SGEMM_OK) rc = SGEMM_ERR_CUDA;
    for (cudaEvent_t ev : {ev_ready, ev_b, ev_done, ev_comp})
        if (ev) cudaEventDestroy(ev);
    for (int c = 0; c < kChunks; ++c) {
        if (ev_a[c]) cudaEventDestroy(ev_a[c]);
        if (ev_p[c]) cudaEventDestroy(ev_p[c]);
        if (ev_c[c]) cudaEventDestroy(ev_c[c]);
    }
    return rc;
}

}  // namespace
}  // namespace sgemm

using namespace sgemm;

namespace {
// cycles over nanoseconds of one kernel's clock record, in MHz
int clock_mhz(cudaError_t (*read)(cudaStream_t, unsigned long long (&)[4]), void* stream,
              double* mhz) {
    if (!mhz) return SGEMM_ERR_ARG;
    int dev = -1;
    if (!current_device(&dev)) return SGEMM_ERR_NO_DEVICE;
    unsigned long long r[4] = {0, 0, 0, 0};
    if (read(static_cast<cudaStream_t>(stream), r) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (r[2] <= r[0] || r[3] <= r[1]) return SGEMM_ERR_UNSUPPORTED;
    *mhz = double(r[3] - r[1]) / double(r[2] - r[0]) * 1e3;
    return SGEMM_OK;
}
}  // namespace

extern "C" {

void solve(const float* A, const float* B, float* C, int M, int N, int K) {
    tl_status = run(A, B, C, M, N, K, SGEMM_MODE_FP32, tl_stream);
}

int solve_ex(const float* A, const float* B, float* C, int M, int N, int K, int mode,
             void* stream) {
    return run(A, B, C, M, N, K, mode, static_cast<cudaStream_t>(stream));
}

int solve_host(const float* hA, const float* hB, float* hC, int M, int N, int K, int mode,
               void* stream_v) {
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_ARG;
    if (!hA || !hB || !hC) return SGEMM_ERR_ARG;
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_3XFP16_SCALED) return SGEMM_ERR_ARG;
    const size_t a_bytes = size_t(M) * N * sizeof(float);
    const size_t b_bytes = size_t(N) * K * sizeof(float);
    const size_t c_bytes = size_t(M) * K * sizeof(float);
    if (ranges_overlap(hC, c_bytes, hA, a_bytes) || ranges_overlap(hC, c_bytes, hB, b_bytes))
        return SGEMM_ERR_OVERLAP;
    int dev = -1;
    const DeviceInfo* info = current_device(&dev);
    if (!info) return SGEMM_ERR_NO_DEVICE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    // Large tensor-core products overlap the copies with the work, chunk by chunk.
    const int kernel = choose_kernel(M, N, K, mode, true);
    if ((kernel == SGEMM_KERNEL_TC_3XTF32 || kernel == SGEMM_KERNEL_TC_1XTF32) && M >= 2048)
        return solve_host_pipelined(hA, hB, hC, M, N, K, kernel == SGEMM_KERNEL_TC_3XTF32 ? 3 : 1,
                                    dev, info, stream);
    int rc = SGEMM_OK;
    {
        Scratch dA, dB, dC;
        if (dA.alloc(dev, a_bytes, stream) != cudaSuccess ||
            dB.alloc(dev, b_bytes, stream) != cudaSuccess ||
            dC.alloc(dev, c_bytes, stream) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        if (cudaMemcpyAsync(dA.ptr, hA, a_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
            cudaMemcpyAsync(dB.ptr, hB, b_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) {
            rc = SGEMM_ERR_CUDA;
        } else {
            rc = run(static_cast<const float*>(dA.ptr), static_cast<const float*>(dB.ptr),
                     static_cast<float*>(dC.ptr), M, N, K, mode, stream);
            if (rc == SGEMM_OK &&
                cudaMemcpyAsync(hC, dC.ptr, c_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
                rc = SGEMM_ERR_CUDA;
        }
    }  // scratch returned to the pool, stream-ordered after the copies
    if (cudaStreamSynchronize(stream) != cudaSuccess && rc == SGEMM_OK) rc = SGEMM_ERR_CUDA;
    return rc;
}

int sgemm_set_stream(void* stream) {
    tl_stream = static_cast<cudaStream_t>(stream);
    return SGEMM_OK;
}

int sgemm_last_status(void) { return tl_status; }

const char* sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK:
            return "ok";
        case SGEMM_ERR_ARG:
            return "invalid argument (dimension outside [1, 8192], null pointer or bad mode)";
        case SGEMM_ERR_OVERLAP:
            return "output C overlaps input A or B";
        case SGEMM_ERR_CUDA:
            return "a CUDA runtime call failed";
        case SGEMM_ERR_NO_DEVICE:
            return "no usable sm_103 CUDA device is current";
        case SGEMM_ERR_TIMEOUT:
            return "a bounded wait inside a kernel gave up";
        case SGEMM_ERR_UNSUPPORTED:
            return "the selected mode cannot serve this shape";
        default:
            return "unknown status";
    }
}

int sgemm_device_error(void* stream) {
    int dev = -1;
    const DeviceInfo* info = current_device(&dev);
    if (!info) return SGEMM_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int word = 0;
    if (cudaMemcpyAsync(&word, info->error_word, sizeof(int), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemsetAsync(info->error_word, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return word == kErrNone ? SGEMM_OK : SGEMM_ERR_TIMEOUT;
}

int sgemm_plan(int M, int N, int K, int mode, int aligned, int* tiles) {
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_ARG;
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_3XFP16_SCALED) return SGEMM_ERR_ARG;
    const int kernel = choose_kernel(M, N, K, mode, aligned != 0);
    if (kernel > 0 && tiles) *tiles = tiles_for(kernel, M, K, aligned && N % 4 == 0 && K % 4 == 0);
    return kernel;
}

int sgemm_plan_units(int M, int N, int K, int mode, int sm_count, int* units, int cap) {
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_ARG;
    if (mode < SGEMM_MODE_FP32 || mode > SGEMM_MODE_3XFP16_SCALED) return SGEMM_ERR_ARG;
    if (sm_count < 0 || sm_count > 1024 || cap < 0 || (cap > 0 && !units)) return SGEMM_ERR_ARG;
    const int sms = sm_count > 0 ? sm_count : 152;
    if (mode == SGEMM_MODE_3XFP16_SCALED) return tc16_schedule_units(M, N, K, sms, units, cap);
    return tc_schedule_units(M, N, K, mode == SGEMM_MODE_TF32 ? 1 : 3, sms, units, cap);
}

long long sgemm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int sgemm_set_kernel_events(void* start, void* stop) {
    tl_ev_start = static_cast<cudaEvent_t>(start);
    tl_ev_stop = static_cast<cudaEvent_t>(stop);
    return SGEMM_OK;
}

int sgemm_selftest_wait_timeout(long long limit_ns, void* stream) {
    if (limit_ns < 1000000 || limit_ns > 2000000000) return SGEMM_ERR_ARG;
    int dev = -1;
    const DeviceInfo* info = current_device(&dev);
    if (!info) return SGEMM_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_wait_selftest(limit_ns, info->error_word, s) != cudaSuccess) return SGEMM_ERR_CUDA;
    return sgemm_device_error(stream);
}

int sgemm_peak_probe(int probe, int iters, void* stream, double* flop, float* ms) {
    if (!flop || !ms || iters < 1) return SGEMM_ERR_ARG;
    if (probe == SGEMM_PROBE_TF32_MMA || probe == SGEMM_PROBE_F16_MMA ? iters > (1 << 18)
                                      : (probe != SGEMM_PROBE_FFMA && probe != SGEMM_PROBE_FFMA2) ||
                                            iters > (1 << 20))
        return SGEMM_ERR_ARG;
    int dev = -1;
    const DeviceInfo* info = current_device(&dev);
    if (!info) return SGEMM_ERR_NO_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    KernelTimer t;
    t.stream = s;
    if (cudaEventCreate(&t.start) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (cudaEventCreate(&t.stop) != cudaSuccess) {
        cudaEventDestroy(t.start);
        return SGEMM_ERR_CUDA;
    }
    cudaError_t e;
    double f;
    if (probe == SGEMM_PROBE_TF32_MMA || probe == SGEMM_PROBE_F16_MMA) {
        const bool f16 = probe == SGEMM_PROBE_F16_MMA;
        e = launch_mma_probe(f16, iters, info->sm_count, info->error_word, s, t);
        f = mma_probe_flops(f16, iters, info->sm_count);
    } else {
        e = launch_ffma_probe(probe == SGEMM_PROBE_FFMA2, iters, info->sm_count, s, t);
        f = ffma_probe_flops(iters, info->sm_count);
    }
    float elapsed = 0.0f;
    if (e == cudaSuccess) e = cudaEventSynchronize(t.stop);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&elapsed, t.start, t.stop);
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
    if (e != cudaSuccess) return SGEMM_ERR_CUDA;
    const int dev_status = sgemm_device_error(stream);
    if (dev_status != SGEMM_OK) return dev_status;
    *flop = f;
    *ms = elapsed;
    return SGEMM_OK;
}

int sgemm_tc_clock_mhz(void* stream, double* mhz) { return clock_mhz(tc_clock_record, stream, mhz); }

int sgemm_simt_clock_mhz(void* stream, double* mhz) {
    return clock_mhz(simt_clock_record, stream, mhz);
}

int sgemm_release_pool(void) {
    int dev = -1;
    if (!current_device(&dev)) return SGEMM_ERR_NO_DEVICE;
    cudaMemPool_t pool;
    if (pool_for(dev, &pool) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
    return cudaMemPoolTrimTo(pool, 0) == cudaSuccess ? SGEMM_OK : SGEMM_ERR_CUDA;
}

}  // extern "C"
