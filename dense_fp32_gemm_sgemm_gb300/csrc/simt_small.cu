// CUDA-core FP32 GEMM for small products: the arithmetic of simt_gemm.cu (every C[m][k]
// one FP32 accumulator updated by round-to-nearest fused multiply-adds with n ascending,
// the fmaf loop of "CUDA 学习笔记 Matrix Multiplication", section "3. V1"), on tiles small
// enough that a product of a few hundred million multiply-adds still occupies every SM.
//
//  * CTA tile 16 x 64 of C with 64 threads (32 x 64 with 128 threads when rows are not
//    16-byte aligned), a 4 x 4 register tile per thread (rows 4 (t / 16) .. +3, columns
//    4 (t % 16) .. +3), updated by rank-1 steps with the packed FP32 FMA (__ffma2_rn, two
//    independent round-to-nearest FMAs per instruction).
//  * A 4-stage cp.async ring of (A: rows x 16, B: 16 x 64) slices with zero fill past the
//    edges (16-byte copies when A and B rows are 16-byte aligned, 4-byte copies otherwise).
//    A is kept n-contiguous with a 20-float row pitch and read four reduction steps at a
//    time in 128-bit loads; B is kept k-contiguous and read in 128-bit loads.
//  * One launch, no workspace: at 512^3 the three launches of the tensor-core path (operand
//    pre-pass, GEMM, split reduction) cost more than these 134 M multiply-adds.
#include "internal.cuh"
#include "ptx.cuh"

namespace sgemm {
namespace {

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
}

// Measured at 512^3, 640^3, 512 x 2048 x 512 and 1024 x 1024 x 512 against 32 x 64 tiles
// of 128 and 256 threads, 16 x 64 of 128 and 32 x 32 of 128: with 16-byte copies 16 x 64
// tiles of 64 threads were fastest (512^3 12.4 against 14.4 us); with 4-byte copies, whose
// per-thread copy count grows as threads shrink, 32 x 64 of 128 (1000 x 333 x 777: 24.7
// against 30.8 us).
using SmallVec = SmallTile<16, 64, 64>;
using SmallScalar = SmallTile<32, 64, 128>;

}  // namespace

int simt_small_tiles(int M, int K, bool vec) {
    return vec ? ((M + SmallVec::BM - 1) / SmallVec::BM) * ((K + SmallVec::BN - 1) / SmallVec::BN)
               : ((M + SmallScalar::BM - 1) / SmallScalar::BM) *
                     ((K + SmallScalar::BN - 1) / SmallScalar::BN);
}

bool simt_small_suits(int M, int K, int sm_count) {
    // the 128 x 128 kernel leaves most SMs idle below one tile per SM
    const int big_tiles = ((M + kSimtBM - 1) / kSimtBM) * ((K + kSimtBN - 1) / kSimtBN);
    return big_tiles < (sm_count > 0 ? sm_count : 1);
}

cudaError_t launch_simt_small(const float* A, const float* B, float* C, int M, int N, int K,
                              bool vec, cudaStream_t stream, const KernelTimer& timer) {
    timer.before();
    if (vec) {
        const dim3 grid((K + SmallVec::BN - 1) / SmallVec::BN, (M + SmallVec::BM - 1) / SmallVec::BM);
        simt_small_kernel<SmallVec, true><<<grid, SmallVec::T, 0, stream>>>(A, B, C, M, N, K);
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

}  // namespace sgemm
