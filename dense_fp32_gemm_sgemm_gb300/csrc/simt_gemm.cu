// CUDA-core FP32 GEMM (FFMA), any shape 1 <= M, N, K <= 8192.
//
// What it computes is the inner-product definition of "LeetGPU |
// 02_Matrix_Multiplication", section "CUDA / Approach": every C[m][k] is one FP32
// accumulator updated by fused multiply-adds with n ascending, the arithmetic of the
// fmaf loop in "CUDA 学习笔记 Matrix Multiplication", section "3. V1". The schedule is
// this file's own:
//
//  * CTA tile 128 x 128 of C, 128 threads, an 8 x 16 register tile per thread updated
//    by rank-1 (outer-product) steps, as in the register-tiling sections ("V1:
//    Two-Dimensional Thread Tiling") but with four times the outputs per thread. The updates
//    use the packed FP32 FMA (__ffma2_rn: two independent round-to-nearest FMAs per
//    instruction), which halves the issue slots the FMAs take. Two CTAs share an SM, so
//    one CTA's barriers and copies overlap the other's FMAs (measured against one
//    256-thread CTA of 128 x 256 per SM: 0.8 % faster at 8192 x 6144 x 4096, 12 % at
//    4096^3, whose last wave the smaller tiles fill better).
//  * A 6-stage cp.async ring of (A: 128 x 16, B: 16 x 128) slices (4 stages with 4-byte
//    copies). Full slices of interior tiles are copied without bounds checks. Elements past an
//    edge are zero-filled by the copy itself (src-size 0), the rule of "V1: Original
//    16 x 16 Shared-Memory Tiling" and "V4: Hardware-Asynchronous cp.async Pipeline".
//    16-byte copies when A/B rows are 16-byte aligned, 4-byte copies otherwise, so
//    unaligned shapes run the same pipeline instead of a scalar fallback.
//  * A is kept n-contiguous in shared memory with a 20-float row pitch, so the 8 rows
//    a warp reads in one 128-bit load fall in 8 disjoint bank quads; B is kept
//    k-contiguous and read as four 128-bit broadcasts per step.
//  * Tiles are visited in groups of 8 tile-rows so that CTAs running together share
//    A and B slices in L2 (the grouped program order of the "Triton" section).
//
// Products too small to fill the SMs with 128 x 128 tiles run on smaller tiles instead
// (simt_split_kernel, which splits the reduction in four inside the CTA, and
// simt_small_kernel, further down).
//
// Integer-valued inputs whose partial sums stay below 2^24 give exact results: every
// product and every partial sum is representable.
#include "internal.cuh"
#include "ptx.cuh"

namespace sgemm {
namespace {

constexpr int BM = kSimtBM;
constexpr int BN = kSimtBN;
constexpr int THREADS = 128;
constexpr int TM = 8;                    // rows per thread: row_base + 8 i, i < TM
constexpr int NJ = 4;                    // groups of 4 columns per thread (TM x 4 NJ register tile)
constexpr int WARPS_M = BM / (8 * TM);   // warps down the tile, 8 TM rows each
constexpr int WARPS_N = BN / (16 * NJ);  // warps across, 16 NJ columns each
constexpr int BK = 16;
// cp.async ring depth: 6 stages for 16-byte copies, 4 for the 4-byte path (measured: the
// deeper ring is 1.5 % faster with 16-byte copies and 0.6 % slower with 4-byte ones)
template <bool VEC>
constexpr int STAGES = VEC ? 6 : 4;
constexpr int A_PITCH = BK + 4;
constexpr int B_PITCH = BN;
constexpr int A_STAGE = BM * A_PITCH;
constexpr int B_STAGE = BK * B_PITCH;
template <bool VEC>
constexpr int SMEM_BYTES = STAGES<VEC> * (A_STAGE + B_STAGE) * int(sizeof(float));
constexpr int GROUP_M = 8;

static_assert(BM == 128 && (BN == 128 || BN == 256) && (BK == 16 || BK == 32) &&
                  (THREADS == 128 || THREADS == 256 || THREADS == 512) && WARPS_M * WARPS_N * 32 == THREADS,
              "index arithmetic below assumes this tiling");

// Interior stage of an interior tile (every row, column and reduction index of the slice
// inside the matrices, rows 16-byte aligned): no bounds checks. The sources are this
// thread's first A and B chunks (a0, b0, at reduction index 0) advanced by the slice's
// reduction offset n0; the thread's further chunks lie a fixed number of rows below.
__device__ __forceinline__ void load_stage_interior(float* As, float* Bs, const float* a0,
                                                    const float* b0, int N, int K, int n0,
                                                    int tid) {
    constexpr int A_ROWS_PER_PASS = THREADS / (BK / 4);
    constexpr int B_ROWS_PER_PASS = THREADS / (BN / 4);
    const int arow = tid / (BK / 4), akc = (tid % (BK / 4)) * 4;
    const int brow = tid / (BN / 4), bcc = (tid % (BN / 4)) * 4;
#pragma unroll
    for (int i = 0; i < BM * BK / 4 / THREADS; ++i)
        ptx::cp_async_16(ptx::smem_u32(As + (arow + i * A_ROWS_PER_PASS) * A_PITCH + akc),
                         a0 + size_t(i * A_ROWS_PER_PASS) * N + n0, true);
    const float* b = b0 + size_t(n0) * K;
#pragma unroll
    for (int i = 0; i < BK * BN / 4 / THREADS; ++i)
        ptx::cp_async_16(ptx::smem_u32(Bs + (brow + i * B_ROWS_PER_PASS) * B_PITCH + bcc),
                         b + size_t(i * B_ROWS_PER_PASS) * K, true);
}

template <bool VEC>
__device__ __forceinline__ void load_stage(float* As, float* Bs, const float* __restrict__ A,
                                           const float* __restrict__ B, int M, int N, int K,
                                           int m0, int k0, int n0, int tid) {
    if constexpr (VEC) {
        // A slice: 128 rows x BK floats, BK / 4 chunks of 16 bytes per row.
#pragma unroll
        for (int i = 0; i < BM * BK / 4 / THREADS; ++i) {
            const int c = tid + i * THREADS;
            const int row = c / (BK / 4), kc = (c % (BK / 4)) * 4;
            const int gm = m0 + row, gn = n0 + kc;
            const bool ok = gm < M && gn < N;
            const float* src = ok ? A + (size_t)gm * N + gn : A;
            ptx::cp_async_16(ptx::smem_u32(As + row * A_PITCH + kc), src, ok);
        }
        // B slice: BK rows x BN floats, BN / 4 chunks per row.
#pragma unroll
        for (int i = 0; i < BK * BN / 4 / THREADS; ++i) {
            const int c = tid + i * THREADS;
            const int row = c / (BN / 4), cc = (c % (BN / 4)) * 4;
            const int gn = n0 + row, gk = k0 + cc;
            const bool ok = gn < N && gk < K;
            const float* src = ok ? B + (size_t)gn * K + gk : B;
            ptx::cp_async_16(ptx::smem_u32(Bs + row * B_PITCH + cc), src, ok);
        }
    } else {
#pragma unroll
        for (int i = 0; i < BM * BK / THREADS; ++i) {
            const int c = tid + i * THREADS;
            const int row = c / BK, kk = c % BK;
            const int gm = m0 + row, gn = n0 + kk;
            const bool ok = gm < M && gn < N;
            const float* src = ok ? A + (size_t)gm * N + gn : A;
            ptx::cp_async_4(ptx::smem_u32(As + row * A_PITCH + kk), src, ok);
        }
#pragma unroll
        for (int i = 0; i < BK * BN / THREADS; ++i) {
            const int c = tid + i * THREADS;
            const int row = c / BN, col = c % BN;
            const int gn = n0 + row, gk = k0 + col;
            const bool ok = gn < N && gk < K;
            const float* src = ok ? B + (size_t)gn * K + gk : B;
            ptx::cp_async_4(ptx::smem_u32(Bs + row * B_PITCH + col), src, ok);
        }
    }
}

__device__ __forceinline__ float lane_of(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// The SM clock the CUDA-core kernels run at: thread 0 of CTA 0 records globaltimer
// nanoseconds and its SM's clock64 cycles when it starts ([0], [1]) and when it ends
// ([2], [3]); the host reads the last launch's record.
__device__ unsigned long long g_simt_clock_record[4];

__device__ __forceinline__ void clock_mark(int end) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        g_simt_clock_record[2 * end] = ptx::globaltimer_ns();
        g_simt_clock_record[2 * end + 1] = clock64();
    }
}

template <bool VEC>
__global__ void __launch_bounds__(THREADS, 1)
    simt_gemm_kernel(const float* __restrict__ A, const float* __restrict__ B,
                     float* __restrict__ C, int M, int N, int K, int tiles_m, int tiles_n) {
    extern __shared__ __align__(16) float smem[];
    clock_mark(0);
    float* As = smem;
    constexpr int S = STAGES<VEC>;
    float* Bs = smem + S * A_STAGE;

    // Grouped tile order: GROUP_M tile-rows at a time, walking down columns.
    const int bid = blockIdx.x;
    const int group_tiles = GROUP_M * tiles_n;
    const int group = bid / group_tiles;
    const int first_m = group * GROUP_M;
    const int rows_in_group = min(GROUP_M, tiles_m - first_m);
    const int in_group = bid - group * group_tiles;
    const int tile_m = first_m + in_group % rows_in_group;
    const int tile_n = in_group / rows_in_group;
    const int m0 = tile_m * BM;
    const int k0 = tile_n * BN;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = (warp / WARPS_N) * (8 * TM);
    const int wn = (warp % WARPS_N) * (16 * NJ);
    const int row_base = wm + (lane >> 2);  // this thread's rows: row_base + 8 i
    const int colq = wn + (lane & 3) * 4;   // and columns colq + 16 j .. +3, j < NJ

    // acc[i][jj]: row i of the thread's TM rows, columns 2 jj and 2 jj + 1 of its 4 NJ
    float2 acc[TM][2 * NJ];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int jj = 0; jj < 2 * NJ; ++jj) acc[i][jj] = make_float2(0.0f, 0.0f);

    const int ktiles = (N + BK - 1) / BK;
    // interior tiles of a 16-byte-aligned product load their full slices without checks
    const int full_ktiles = VEC && m0 + BM <= M && k0 + BN <= K ? N / BK : 0;
    const float* a0 = A + size_t(m0 + tid / (BK / 4)) * N + (tid % (BK / 4)) * 4;
    const float* b0 = B + size_t(tid / (BN / 4)) * K + k0 + (tid % (BN / 4)) * 4;
    auto load = [&](int t) {
        float* as_t = As + (t % S) * A_STAGE;
        float* bs_t = Bs + (t % S) * B_STAGE;
        if (t < full_ktiles)
            load_stage_interior(as_t, bs_t, a0, b0, N, K, t * BK, tid);
        else
            load_stage<VEC>(as_t, bs_t, A, B, M, N, K, m0, k0, t * BK, tid);
    };
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        if (s < ktiles) load(s);
        ptx::cp_async_commit();
    }

    for (int kt = 0; kt < ktiles; ++kt) {
        ptx::cp_async_wait<S - 2>();
        __syncthreads();
        const int nt = kt + S - 1;
        if (nt < ktiles) load(nt);
        ptx::cp_async_commit();

        const float* as = As + (kt % S) * A_STAGE;
        const float* bs = Bs + (kt % S) * B_STAGE;
#pragma unroll
        for (int kc = 0; kc < BK; kc += 4) {
            float4 a[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = *reinterpret_cast<const float4*>(as + (row_base + 8 * i) * A_PITCH + kc);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float2 bp[2 * NJ];
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const float4 b =
                        *reinterpret_cast<const float4*>(bs + (kc + kk) * B_PITCH + colq + 16 * j);
                    bp[2 * j] = make_float2(b.x, b.y);
                    bp[2 * j + 1] = make_float2(b.z, b.w);
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float av = lane_of(a[i], kk);
                    const float2 a2 = make_float2(av, av);
                    // two independent round-to-nearest FMAs per instruction (the packed
                    // FP32 FMA of sm_100+), the same arithmetic as fmaf per element
#pragma unroll
                    for (int jj = 0; jj < 2 * NJ; ++jj)
                        acc[i][jj] = __ffma2_rn(a2, bp[jj], acc[i][jj]);
                }
            }
        }
    }
    ptx::cp_async_wait<0>();

    // Epilogue: registers -> C, 128-bit stores when rows are 16-byte aligned.
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + row_base + 8 * i;
        if (row >= M) continue;
        float* crow = C + (size_t)row * K;
#pragma unroll
        for (int h = 0; h < NJ; ++h) {
            const int col = k0 + colq + 16 * h;
            const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                acc[i][2 * h + 1].y};
            if constexpr (VEC) {
                if (col < K)
                    *reinterpret_cast<float4*>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < K) crow[col + j] = v[j];
            }
        }
    }
    clock_mark(1);
}

template <bool VEC>
cudaError_t launch_impl(const float* A, const float* B, float* C, int M, int N, int K,
                        cudaStream_t stream, const KernelTimer& timer) {
    cudaError_t err = set_smem_limit_once<simt_gemm_kernel<VEC>>(SMEM_BYTES<VEC>);
    if (err != cudaSuccess) return err;
    const int tiles_m = (M + BM - 1) / BM;
    const int tiles_n = (K + BN - 1) / BN;
    timer.before();
    simt_gemm_kernel<VEC><<<tiles_m * tiles_n, THREADS, SMEM_BYTES<VEC>, stream>>>(A, B, C, M, N, K,
                                                                             tiles_m, tiles_n);
    err = cudaGetLastError();
    timer.after();
    count_launch();
    return err;
}

// Rate probe for the FP32 FMA pipe: each thread runs 16 independent chains of
// x <- x * s + t (s, t chosen at run time), as scalar fmaf or as eight packed
// __ffma2_rn, with no memory traffic in the loop. The sums are compared with a value they
// cannot take, so the chains are kept without storing them.
__device__ float g_probe_sink;

template <bool PACKED>
__global__ void __launch_bounds__(256) ffma_probe_kernel(int iters, float s, float t) {
    clock_mark(0);
    float r = 0.0f;
    if constexpr (PACKED) {
        float2 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = make_float2(threadIdx.x * 1e-3f + j, 0.5f * j);
        const float2 s2 = make_float2(s, s), t2 = make_float2(t, t);
#pragma unroll 4
        for (int i = 0; i < iters; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = __ffma2_rn(x[j], s2, t2);
#pragma unroll
        for (int j = 0; j < 8; ++j) r += x[j].x + x[j].y;
    } else {
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = threadIdx.x * 1e-3f + j;
#pragma unroll 4
        for (int i = 0; i < iters; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = fmaf(x[j], s, t);
#pragma unroll
        for (int j = 0; j < 16; ++j) r += x[j];
    }
    if (r == t * 1.0e30f) g_probe_sink = r;
    clock_mark(1);
}

constexpr int kProbeBlocksPerSm = 8;

// ----------------------------------------------------- small products (FFMA) ------
// Small products run on tiles small enough that a product of a few hundred million
// multiply-adds still occupies every SM, in one launch with no workspace (at 512^3 the
// three launches of the tensor-core path, operand pre-pass, GEMM and split reduction,
// cost more than these 134 M multiply-adds).
//
// 16-byte aligned rows (simt_split_kernel): the reduction is split inside the CTA.
//  * CTA tile 16 x 64 of C (16 x 32 when 16 x 64 tiles would leave SMs idle), four groups
//    of 32 threads. Each stage holds 64 reduction elements; group g multiplies elements
//    [16 g, 16 g + 16) of every stage, so each C[m][k] is the sum of four FP32
//    accumulators, each updated by round-to-nearest fused multiply-adds with n ascending
//    over its slices, added in group order at the end ((acc0 + acc1) + acc2) + acc3
//    through shared memory. Four times the threads of an unsplit tile, each with a
//    quarter of the serial multiply-add chain: at 512^3 9.5 against 11.2 us of device
//    time for the unsplit 16 x 64 kernel, at 256^3 3.2 against 5.7 us.
//  * A thread owns a 4 x 8 block of the 16 x 64 tile (4 x 4 of the 16 x 32 tile): rows
//    4 (t / CQ) .. +3 and the 4-column quads t % CQ and t % CQ + CQ (CQ quads per half
//    row, so a warp's B loads are contiguous), updated by rank-1 steps with the packed
//    FP32 FMA (__ffma2_rn). Wider thread blocks (1 x 16, 2 x 8) measured slower: each
//    128-bit shared-memory load feeds fewer multiply-adds.
//  * A 2-stage cp.async ring with zero fill past the edges; A n-contiguous with a row
//    pitch of 68 floats, B k-contiguous.
// Rows that are not 16-byte aligned (simt_small_kernel): CTA tile 32 x 64, 128 threads,
// a 4 x 4 register tile per thread (rows 4 (t / 16) .. +3, columns 4 (t % 16) .. +3), one
// accumulator per element with n ascending, and a 4-stage ring of 4-byte copies.
constexpr int SBK = 16;   // reduction elements per stage
constexpr int SSTAGES = 4;
constexpr int SA_PITCH = SBK + 4;

// Tile BM_ x BN_ of C per CTA, T_ threads, each thread TM rows x 4 columns.
template <int BM_, int BN_, int T_>
struct SmallTile {
    static constexpr int BM = BM_, BN = BN_, T = T_;
    static constexpr int TM = BM * BN / (4 * T);      // rows per thread
    static constexpr int CG = BN / 4;                 // column groups of 4
    static constexpr int A_STAGE = BM * SA_PITCH;
    static constexpr int B_STAGE = SBK * BN;
    static constexpr int A_CHUNKS = BM * SBK / 4;     // 16-byte chunks per stage
    static constexpr int B_CHUNKS = SBK * BN / 4;
    static_assert(TM >= 1 && TM * 4 * T == BM * BN && T % CG == 0 && (T / CG) * TM == BM,
                  "each thread a TM x 4 block, threads tile the CTA tile exactly");
    static_assert(B_CHUNKS % T == 0 && (A_CHUNKS % T == 0 || T % A_CHUNKS == 0), "chunk split");
};

// One stage: A rows [m0, m0 + BM) x reduction [n0, n0 + 16), B reduction rows
// [n0, n0 + 16) x columns [k0, k0 + BN); elements outside the matrices are zero.
template <class TL, bool VEC>
__device__ __forceinline__ void load_small_stage(float* As, float* Bs, const float* __restrict__ A,
                                                 const float* __restrict__ B, int M, int N, int K,
                                                 int m0, int k0, int n0, int tid) {
    if constexpr (VEC) {
#pragma unroll
        for (int c = tid; c < TL::A_CHUNKS; c += TL::T) {
            const int row = c / (SBK / 4), kc = (c % (SBK / 4)) * 4;
            const int gm = m0 + row, gn = n0 + kc;
            const bool ok = gm < M && gn < N;  // N % 4 == 0: the chunk is whole or outside
            ptx::cp_async_16(ptx::smem_u32(As + row * SA_PITCH + kc),
                             ok ? A + size_t(gm) * N + gn : A, ok);
        }
#pragma unroll
        for (int c = tid; c < TL::B_CHUNKS; c += TL::T) {
            const int row = c / TL::CG, cc = (c % TL::CG) * 4;
            const int gn = n0 + row, gk = k0 + cc;
            const bool ok = gn < N && gk < K;  // K % 4 == 0
            ptx::cp_async_16(ptx::smem_u32(Bs + row * TL::BN + cc),
                             ok ? B + size_t(gn) * K + gk : B, ok);
        }
    } else {
#pragma unroll
        for (int c = tid; c < TL::BM * SBK; c += TL::T) {
            const int row = c / SBK, kk = c % SBK;
            const int gm = m0 + row, gn = n0 + kk;
            const bool ok = gm < M && gn < N;
            ptx::cp_async_4(ptx::smem_u32(As + row * SA_PITCH + kk),
                            ok ? A + size_t(gm) * N + gn : A, ok);
        }
#pragma unroll
        for (int c = tid; c < SBK * TL::BN; c += TL::T) {
            const int row = c / TL::BN, col = c % TL::BN;
            const int gn = n0 + row, gk = k0 + col;
            const bool ok = gn < N && gk < K;
            ptx::cp_async_4(ptx::smem_u32(Bs + row * TL::BN + col),
                            ok ? B + size_t(gn) * K + gk : B, ok);
        }
    }
}

__device__ __forceinline__ float lane4(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <class TL, bool VEC>
__global__ void __launch_bounds__(TL::T)
    simt_small_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K) {
    constexpr int TM = TL::TM;
    __shared__ __align__(16) float As[SSTAGES * TL::A_STAGE];
    __shared__ __align__(16) float Bs[SSTAGES * TL::B_STAGE];
    clock_mark(0);
    const int tid = threadIdx.x;
    const int m0 = int(blockIdx.y) * TL::BM, k0 = int(blockIdx.x) * TL::BN;
    const int r0 = (tid / TL::CG) * TM, c0 = (tid % TL::CG) * 4;  // this thread's block

    // acc[i][h]: row r0 + i, columns c0 + 2 h and c0 + 2 h + 1
    float2 acc[TM][2];
#pragma unroll
    for (int i = 0; i < TM; ++i) acc[i][0] = acc[i][1] = make_float2(0.0f, 0.0f);

    const int ktiles = (N + SBK - 1) / SBK;
#pragma unroll
    for (int s = 0; s < SSTAGES - 1; ++s) {
        if (s < ktiles)
            load_small_stage<TL, VEC>(As + s * TL::A_STAGE, Bs + s * TL::B_STAGE, A, B, M, N, K,
                                      m0, k0, s * SBK, tid);
        ptx::cp_async_commit();
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        ptx::cp_async_wait<SSTAGES - 2>();
        __syncthreads();
        const int nt = kt + SSTAGES - 1;
        if (nt < ktiles)
            load_small_stage<TL, VEC>(As + (nt % SSTAGES) * TL::A_STAGE,
                                      Bs + (nt % SSTAGES) * TL::B_STAGE, A, B, M, N, K, m0, k0,
                                      nt * SBK, tid);
        ptx::cp_async_commit();
        const float* as = As + (kt % SSTAGES) * TL::A_STAGE;
        const float* bs = Bs + (kt % SSTAGES) * TL::B_STAGE;
#pragma unroll
        for (int kc = 0; kc < SBK; kc += 4) {
            float4 a[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = *reinterpret_cast<const float4*>(as + (r0 + i) * SA_PITCH + kc);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 b = *reinterpret_cast<const float4*>(bs + (kc + kk) * TL::BN + c0);
                const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float av = lane4(a[i], kk);
                    const float2 a2 = make_float2(av, av);
                    acc[i][0] = __ffma2_rn(a2, b01, acc[i][0]);
                    acc[i][1] = __ffma2_rn(a2, b23, acc[i][1]);
                }
            }
        }
    }
    ptx::cp_async_wait<0>();

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int row = m0 + r0 + i;
        const int col = k0 + c0;
        if (row >= M || col >= K) continue;
        float* dst = C + size_t(row) * K + col;
        if constexpr (VEC) {
            *reinterpret_cast<float4*>(dst) =  // K % 4 == 0: the 4 columns are inside
                make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
        } else {
            const float v[4] = {acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < K) dst[j] = v[j];
        }
    }
    clock_mark(1);
}

using SmallScalar = SmallTile<32, 64, 128>;

// Split-reduction tile: BM x BN of C, S groups of T threads, each thread TM rows x TN
// columns (TN / 4 quads, BN / (TN / 4) apart).
constexpr int SPLIT_S = 4;
constexpr int SPLIT_STAGES = 2;
template <int BM_, int BN_, int TM_, int TN_>
struct SplitTile {
    static constexpr int BM = BM_, BN = BN_, TM = TM_, TN = TN_, S = SPLIT_S;
    static constexpr int Q = TN / 4;                  // column quads per thread
    static constexpr int CQ = BN / TN;                // quad positions per BN / Q columns
    static constexpr int T = (BM / TM) * CQ;          // threads per group
    static constexpr int D = SBK * S;                 // reduction elements per stage
    static constexpr int A_PITCH = D + 4;
    static constexpr int A_STAGE = BM * A_PITCH;
    static constexpr int B_STAGE = D * BN;
    static constexpr int FLOATS = SPLIT_STAGES * (A_STAGE + B_STAGE);
    static_assert(T * TM * TN == BM * BN && BN % TN == 0 && TN % 4 == 0, "threads tile the CTA tile");
    static_assert((S - 1) * BM * BN <= FLOATS, "the partial tiles fit in the ring");
};
using SplitWide = SplitTile<16, 64, 4, 8>;    // 32 threads per group, 128 per CTA
using SplitNarrow = SplitTile<16, 32, 4, 4>;  // 32 threads per group, 128 per CTA

template <class TL>
__global__ void __launch_bounds__(TL::T * TL::S)
    simt_split_kernel(const float* __restrict__ A, const float* __restrict__ B,
                      float* __restrict__ C, int M, int N, int K) {
    constexpr int TM = TL::TM, Q = TL::Q, D = TL::D, AP = TL::A_PITCH;
    constexpr int NT = TL::T * TL::S;
    __shared__ __align__(16) float sm[TL::FLOATS];
    float* As = sm;
    float* Bs = sm + SPLIT_STAGES * TL::A_STAGE;
    clock_mark(0);
    const int tid = threadIdx.x, g = tid / TL::T, t = tid % TL::T;
    const int m0 = int(blockIdx.y) * TL::BM, k0 = int(blockIdx.x) * TL::BN;
    const int r0 = (t / TL::CQ) * TM, c0 = (t % TL::CQ) * 4;  // quads c0 + q BN / Q

    // acc[i][2 q + h]: row r0 + i, columns c0 + q BN / Q + 2 h, + 1
    float2 acc[TM][2 * Q];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 2 * Q; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    // stage: A rows [m0, m0 + BM) x reduction [n0, n0 + D), B rows [n0, n0 + D) x columns
    // [k0, k0 + BN), 16-byte copies (N % 4 == 0 and K % 4 == 0: a chunk is whole or
    // outside), zero past the edges
    auto load = [&](int st, int n0) {
        float* as = As + st * TL::A_STAGE;
        float* bs = Bs + st * TL::B_STAGE;
#pragma unroll
        for (int c = tid; c < TL::BM * D / 4; c += NT) {
            const int row = c / (D / 4), kc = (c % (D / 4)) * 4;
            const int gm = m0 + row, gn = n0 + kc;
            const bool ok = gm < M && gn < N;
            ptx::cp_async_16(ptx::smem_u32(as + row * AP + kc), ok ? A + size_t(gm) * N + gn : A, ok);
        }
#pragma unroll
        for (int c = tid; c < D * TL::BN / 4; c += NT) {
            const int row = c / (TL::BN / 4), cc = (c % (TL::BN / 4)) * 4;
            const int gn = n0 + row, gk = k0 + cc;
            const bool ok = gn < N && gk < K;
            ptx::cp_async_16(ptx::smem_u32(bs + row * TL::BN + cc), ok ? B + size_t(gn) * K + gk : B,
                             ok);
        }
    };

    const int ktiles = (N + D - 1) / D;
    load(0, 0);
    ptx::cp_async_commit();
    for (int kt = 0; kt < ktiles; ++kt) {
        ptx::cp_async_wait<0>();
        __syncthreads();  // stage kt is in; every group is done with stage kt - 1
        if (kt + 1 < ktiles) load((kt + 1) % SPLIT_STAGES, (kt + 1) * D);
        ptx::cp_async_commit();
        const float* as = As + (kt % SPLIT_STAGES) * TL::A_STAGE + g * SBK;
        const float* bs = Bs + (kt % SPLIT_STAGES) * TL::B_STAGE + g * SBK * TL::BN;
#pragma unroll
        for (int kc = 0; kc < SBK; kc += 4) {
            float4 a[TM];
#pragma unroll
            for (int i = 0; i < TM; ++i)
                a[i] = *reinterpret_cast<const float4*>(as + (r0 + i) * AP + kc);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float2 bp[2 * Q];
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const float4 b = *reinterpret_cast<const float4*>(
                        bs + (kc + kk) * TL::BN + c0 + q * (TL::BN / Q));
                    bp[2 * q] = make_float2(b.x, b.y);
                    bp[2 * q + 1] = make_float2(b.z, b.w);
                }
#pragma unroll
                for (int i = 0; i < TM; ++i) {
                    const float av = lane4(a[i], kk);
                    const float2 a2 = make_float2(av, av);
#pragma unroll
                    for (int j = 0; j < 2 * Q; ++j) acc[i][j] = __ffma2_rn(a2, bp[j], acc[i][j]);
                }
            }
        }
    }
    ptx::cp_async_wait<0>();
    __syncthreads();  // every group is done reading the ring

    // groups 1 .. S-1 park their partial tiles in the ring; group 0 adds them in order
    float* part = sm;
    if (g > 0) {
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int q = 0; q < Q; ++q)
                *reinterpret_cast<float4*>(part + ((g - 1) * TL::BM + r0 + i) * TL::BN + c0 +
                                           q * (TL::BN / Q)) =
                    make_float4(acc[i][2 * q].x, acc[i][2 * q].y, acc[i][2 * q + 1].x,
                                acc[i][2 * q + 1].y);
    }
    __syncthreads();
    if (g == 0) {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int row = m0 + r0 + i;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int cl = c0 + q * (TL::BN / Q);
                float4 v = make_float4(acc[i][2 * q].x, acc[i][2 * q].y, acc[i][2 * q + 1].x,
                                       acc[i][2 * q + 1].y);
#pragma unroll
                for (int h = 1; h < TL::S; ++h) {
                    const float4 p =
                        *reinterpret_cast<const float4*>(part + ((h - 1) * TL::BM + r0 + i) * TL::BN + cl);
                    v.x += p.x;
                    v.y += p.y;
                    v.z += p.z;
                    v.w += p.w;
                }
                const int col = k0 + cl;
                if (row < M && col < K)  // K % 4 == 0: the 4 columns are inside
                    *reinterpret_cast<float4*>(C + size_t(row) * K + col) = v;
            }
        }
    }
    clock_mark(1);
}

// 16 x 64 tiles unless they would leave SMs idle
bool split_wide(int M, int K, int sm_count) {
    const int tiles = ((M + SplitWide::BM - 1) / SplitWide::BM) * ((K + SplitWide::BN - 1) / SplitWide::BN);
    return tiles >= (sm_count > 0 ? sm_count : 1);
}

}  // namespace

cudaError_t launch_ffma_probe(bool packed, int iters, int sm_count, cudaStream_t stream,
                              const KernelTimer& timer) {
    const int blocks = (sm_count > 0 ? sm_count : 1) * kProbeBlocksPerSm;
    // load the kernel before the start event, so that a lazy module load is not timed
    cudaFuncAttributes attr;
    cudaError_t e = packed ? cudaFuncGetAttributes(&attr, ffma_probe_kernel<true>)
                           : cudaFuncGetAttributes(&attr, ffma_probe_kernel<false>);
    if (e != cudaSuccess) return e;
    timer.before();
    if (packed)
        ffma_probe_kernel<true><<<blocks, THREADS, 0, stream>>>(iters, 0.999f, 1.0e-3f);
    else
        ffma_probe_kernel<false><<<blocks, THREADS, 0, stream>>>(iters, 0.999f, 1.0e-3f);
    e = cudaGetLastError();
    timer.after();
    count_launch();
    return e;
}

double ffma_probe_flops(int iters, int sm_count) {
    const int blocks = (sm_count > 0 ? sm_count : 1) * kProbeBlocksPerSm;
    return double(blocks) * THREADS * iters * 16 * 2.0;
}

cudaError_t launch_simt(const float* A, const float* B, float* C, int M, int N, int K, bool vec,
                        cudaStream_t stream, const KernelTimer& timer) {
    return vec ? launch_impl<true>(A, B, C, M, N, K, stream, timer)
               : launch_impl<false>(A, B, C, M, N, K, stream, timer);
}

int simt_small_tiles(int M, int K, bool vec, int sm_count) {
    if (!vec)
        return ((M + SmallScalar::BM - 1) / SmallScalar::BM) *
               ((K + SmallScalar::BN - 1) / SmallScalar::BN);
    return split_wide(M, K, sm_count)
               ? ((M + SplitWide::BM - 1) / SplitWide::BM) * ((K + SplitWide::BN - 1) / SplitWide::BN)
               : ((M + SplitNarrow::BM - 1) / SplitNarrow::BM) *
                     ((K + SplitNarrow::BN - 1) / SplitNarrow::BN);
}

bool simt_small_suits(int M, int K, int sm_count) {
    // the 128 x 128 kernel leaves most SMs idle below one tile per SM
    const int big_tiles = ((M + kSimtBM - 1) / kSimtBM) * ((K + kSimtBN - 1) / kSimtBN);
    return big_tiles < (sm_count > 0 ? sm_count : 1);
}

cudaError_t launch_simt_small(const float* A, const float* B, float* C, int M, int N, int K,
                              bool vec, int sm_count, cudaStream_t stream, const KernelTimer& timer) {
    timer.before();
    if (vec && split_wide(M, K, sm_count)) {
        const dim3 grid((K + SplitWide::BN - 1) / SplitWide::BN, (M + SplitWide::BM - 1) / SplitWide::BM);
        simt_split_kernel<SplitWide><<<grid, SplitWide::T * SplitWide::S, 0, stream>>>(A, B, C, M, N, K);
    } else if (vec) {
        const dim3 grid((K + SplitNarrow::BN - 1) / SplitNarrow::BN,
                        (M + SplitNarrow::BM - 1) / SplitNarrow::BM);
        simt_split_kernel<SplitNarrow><<<grid, SplitNarrow::T * SplitNarrow::S, 0, stream>>>(A, B, C, M, N,
                                                                                         K);
    } else {
        const dim3 grid((K + SmallScalar::BN - 1) / SmallScalar::BN,
                        (M + SmallScalar::BM - 1) / SmallScalar::BM);
        simt_small_kernel<SmallScalar, false><<<grid, SmallScalar::T, 0, stream>>>(A, B, C, M, N,
                                                                                  K);
    }
    const cudaError_t err = cudaGetLastError();
    timer.after();
    count_launch();
    return err;
}

cudaError_t simt_clock_record(cudaStream_t stream, unsigned long long (&out)[4]) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_simt_clock_record, sizeof(out), 0,
                                              cudaMemcpyDeviceToHost, stream);
    return e == cudaSuccess ? cudaStreamSynchronize(stream) : e;
}

}  // namespace sgemm
