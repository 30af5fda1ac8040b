// Tensor-core (tcgen05) GEMM for sm_103a: one or three TF32 products per term
// (kind::tf32), or three FP16 products of scaled pieces (kind::f16, an explicit mode).
//
// Arithmetic.
//  * 1xTF32: each input is rounded to TF32 with round-to-nearest, ties away from zero
//    (cvt.rna), and the products are accumulated in FP32 - the explicit TF32 path of
//    "LeetGPU | 02_Matrix_Multiplication", section "V5: WMMA TF32 Tensor Core Kernel".
//  * 3xTF32 (FP32-accurate): x = hi + lo with hi = x truncated to TF32 and
//    lo = rna(x - hi) (x - hi is exact in FP32), and A.B ~ A_lo.B_hi + A_hi.B_lo +
//    A_hi.B_hi, the smallest terms first. The tensor core reads a kind::tf32 operand's
//    upper 19 bits and ignores the low 13 (measured: an unrounded A times the identity
//    returns A truncated, bit for bit), so a 16-byte aligned A with rows of a multiple
//    of 4 floats is loaded as its own hi plane and only its lo plane is written. B's hi
//    plane is written anyway (B is transposed) and is written truncated. Each input
//    keeps at least 21 significant bits; the rounding of lo
//    and the dropped A_lo.B_lo term are below 2^-21 + 2^-21 of |a||b| per product (about
//    1e-8 of sum |a||b| on the workloads' inputs, far below the FP32 accumulation
//    error).
//  * 3xFP16 (explicit mode): each row of A and each 128-column block of B is scaled by a
//    power of two that puts its largest magnitude in [2^14, 2^15), split into FP16
//    hi = rn(x) and lo = rn(x - hi), and multiplied as in 3xTF32 with kind::f16 MMAs,
//    which take twice as many elements per clock; the epilogue undoes the scales. An
//    element far below its row's (block's) largest keeps fewer bits (the lo piece leaves
//    FP16's normal range), hence a bound with an absolute term, stated in the header.
//
// Accumulation. The tensor core's FP32 accumulation is not round-to-nearest: measured
// on this part, its error is biased and grows with the number of MMA steps folded into
// one accumulator (about 1e-4 of sum |a||b| after 3 * 8192 / 8 steps on same-sign
// data). The 3xTF32 kernel therefore restarts its TMEM accumulator every SEG_KB
// reduction blocks and adds each segment into FP32 registers with round-to-nearest, so
// the tensor-core error is that of SEG_KB blocks only. The 1xTF32 kernel keeps one
// accumulator per tile: its input rounding (2^-11 per operand) dominates anyway.
//
// Data path.
//  * A pre-pass (tf32_prep_kernel) writes the rounded planes of B transposed (so that
//    both operands are contiguous along the reduction) and of A, to a workspace whose
//    rows are padded to 16-byte multiples. Every shape and every input alignment so
//    reaches the GEMM as TMA-legal tensors; TMA's out-of-bounds zero fill supplies the
//    ragged edges. For a large aligned A the GEMM kernel splits A itself: the first
//    round's rows chunk by chunk before the first MMAs, the rows of later rounds while
//    earlier tiles are multiplied (FusedSplit).
//  * Persistent kernels in clusters of two CTAs (one per SM of a pair). A pair computes
//    256 x 256 output tiles, in grouped order, with tcgen05.mma.cta_group::2 (M=256,
//    N=256, K=8 TF32 or K=16 FP16): each CTA holds 128 rows of A and 128 rows of B^T in
//    its own shared memory, so each SM stages and reads half of the B tile.
//    In each CTA, warp 0 issues TMA loads of its halves into the stage ring (per
//    reduction block of one 128-byte row, 32 floats or 64 halves: the hi planes, 6
//    stages, or the hi and lo planes, 3 stages; 128-row blocks, reduction-contiguous,
//    128-byte swizzled), signalling the leader
//    CTA's barrier; warp 1 of the leader issues the pair MMAs into TMEM (each CTA's TMEM
//    holds its 128 rows of the accumulator) and commits them to barriers in both CTAs;
//    the epilogue warps of both CTAs drain their TMEM with tcgen05.ld and store C
//    through shared memory with TMA tensor stores. Two 256-column TMEM accumulators let
//    the drain overlap the next MMAs. The two products of each 3xTF32 slice that share
//    A_hi take it from the MMA collector buffer the first one fills.
//  * Long 1xTF32 products run on 256 x 512 pair tiles instead (tc_gemm_wide_kernel): a
//    stage then feeds 8 MMAs, the accumulator fills TMEM and is drained once per tile.
//  * CTA 0 records the SM clock it ran at (g_clock_record): under the chip's power
//    limit these kernels run below the maximum clock, and the host reports the rate
//    against the clock actually held.
//  * Every wait is bounded (a few seconds of %globaltimer): a wait that runs out sets
//    the device error word and an abort flag in shared memory, every role leaves its
//    loop, in-flight MMAs are drained, TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <utility>

#include "internal.cuh"
#include "ptx.cuh"

namespace sgemm {
namespace {

constexpr int BM = kTcBM;      // rows of one output tile, computed by a CTA pair
constexpr int BN = kTcBN;      // columns of one output tile
constexpr int HALF_M = BM / 2; // rows of A (and of the tile) held by each CTA of the pair
constexpr int HALF_N = BN / 2; // rows of B^T (output columns) held by each CTA
constexpr int BK = 32;         // floats per stage along the reduction (128 bytes)
constexpr int UMMA_K = 8;  // kind::tf32 consumes 8 elements (32 bytes) of K per MMA
constexpr int A_PLANE_BYTES = HALF_M * BK * 4;  // this CTA's 128 x 32 block of one A plane
constexpr int B_PLANE_BYTES = HALF_N * BK * 4;  // this CTA's 128 x 32 block of one B^T plane
constexpr int RING_BYTES = 6 * (A_PLANE_BYTES + B_PLANE_BYTES);  // 192 KiB of stages
constexpr int MAX_STAGES = 6;
constexpr int TMEM_COLS = 2 * BN;
constexpr int GROUP_M = 8;
constexpr int NUM_BARS = 2 * MAX_STAGES + 4 + 1;
// C staging for the TMA-store epilogue: 32 x 32 float blocks (4 KiB, 128-byte swizzled),
// eight after the ring's 192 KiB plus whatever a shorter ring leaves free, shared out
// evenly among the epilogue warps.
constexpr int STAGING_FIXED = 8;
constexpr int STAGING_BYTES = 32 * 32 * 4;
constexpr int SMEM_BYTES = RING_BYTES + STAGING_FIXED * STAGING_BYTES + 256 + 1024;
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;
// tile-accumulator kernel: TMA warp, MMA warp, 4 epilogue warps (per CTA)
constexpr int THREADS_TILE = 192;
constexpr int EPI_WARPS_TILE = 4;
// with A's split fused into the kernel: four more warps that split rows
constexpr int THREADS_TILE_FUSED = 320;
// segmented kernel: TMA warp, MMA warp, 8 epilogue warps (two per TMEM lane quarter,
// each owning 128 of the 256 columns)
constexpr int THREADS_SEG = 320;
constexpr int EPI_WARPS_SEG = 8;
// with A's split fused into the kernel, two more warps do nothing but split rows (the
// register file allows it: ptxas allocates 320 threads like 384)
constexpr int THREADS_SEG_FUSED = 384;
constexpr int SEG_KB = 4;  // reduction blocks (of BK) per accumulator segment
constexpr int PREP_BT = 64;  // side of the pre-pass's transpose tile of B
constexpr int PREP_A_UNROLL = 4;  // 128-bit loads of A in flight per pre-pass thread
constexpr uint16_t PAIR_MASK = 0x3;

static_assert(BM == 256 && BN == 256, "epilogue and descriptors assume 256 x 256 pair tiles");

// The stage ring. A stage holds, for one reduction block, PLANES_ operand planes of this
// CTA's halves: the hi plane (1xTF32, 6 stages of 32 KiB), or the hi and lo planes
// (3xTF32, 3 stages of 64 KiB), so that each plane block is fetched once per reduction
// block and feeds every MMA that uses it. Layout of a stage: A planes, then B^T planes.
// (A 2-stage 3xTF32 ring, giving its 64 KiB to C staging, was measured on short
// reductions: 4% faster at N = 64, 17-20% slower at N = 128 and 256.)
template <int PLANES_, int STAGES_>
struct Ring {
    static constexpr int PLANES = PLANES_;
    static constexpr int STAGES = STAGES_;
    static constexpr int STAGE_BYTES = PLANES * (A_PLANE_BYTES + B_PLANE_BYTES);
    static constexpr int BYTES = STAGES * STAGE_BYTES;
    static constexpr int STAGING_BLOCKS = (RING_BYTES - BYTES) / STAGING_BYTES + STAGING_FIXED;
    static __device__ __forceinline__ uint32_t a_off(int p) { return uint32_t(p) * A_PLANE_BYTES; }
    static __device__ __forceinline__ uint32_t b_off(int p) {
        return uint32_t(PLANES) * A_PLANE_BYTES + uint32_t(p) * B_PLANE_BYTES;
    }
    static_assert(STAGES >= 2 && STAGES <= MAX_STAGES && BYTES <= RING_BYTES, "ring sizing");
};
using Ring1 = Ring<1, 6>;  // 1xTF32: two staging blocks per epilogue warp
using Ring3 = Ring<2, 3>;  // 3xTF32: one staging block per epilogue warp
static_assert(Ring1::STAGING_BLOCKS == 8 && Ring3::STAGING_BLOCKS == 8, "staging sizing");
static_assert(BK * 4 == 128, "one stage row must be one 128-byte swizzle row");

// ---------------------------------------------------------------- descriptors ------
// Shared-memory matrix descriptor (tcgen05): start address, leading and stride byte
// offsets (all >> 4), descriptor version 1 at bit 46, 128-byte swizzle (value 2) in
// bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor for kind::tf32: FP32 accumulator (bits 4-5 = 1), A and B TF32
// (bits 7-9 and 10-12 = 2), both K-major (bits 15 and 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28. For a CTA pair M and N are the pair's totals (256 x 256).
__host__ __device__ constexpr uint32_t idesc_tf32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(n >> 3) << 17) |
           (uint32_t(m >> 4) << 24);
}
// kind::f16 with FP16 A and B (format 0 in both fields) and an FP32 accumulator
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
    return (1u << 4) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}
// Reduction elements in one 128-byte row of a stage: 32 floats, or 64 halves (FP16 planes).
template <bool F16>
constexpr int BK_ELEMS = F16 ? 64 : 32;
// Columns of B that share one power-of-two scale in the FP16 path (a multiple of 32, so a
// warp's columns never straddle two blocks)
constexpr int F16_COL_BLOCK = 128;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The SM clock the tensor-core kernels run at: CTA 0 of each GEMM (and of the rate probe)
// records globaltimer nanoseconds and its SM's clock64 cycles when its first MMA is
// issued ([0], [1]) and when its last result is stored ([2], [3]). The last launch's
// record is read back by the host; it costs four stores per launch.
__device__ unsigned long long g_clock_record[4];

__device__ __forceinline__ void clock_mark(int end) {
    if (blockIdx.x == 0) {
        g_clock_record[2 * end] = global_ns();
        g_clock_record[2 * end + 1] = clock64();
    }
}

// Waits for the barrier phase of the given parity (acquire at cluster scope when
// `cluster` is set: the barrier is signalled from the peer CTA). Returns false if the
// wait ran out of time (then it raises the abort flag and the device error word) or if
// another role of this CTA already aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err,
                                           unsigned long long limit_ns = WAIT_LIMIT_NS,
                                           bool cluster = false) {
    auto probe = [&]() {
        return cluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (probe()) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (probe()) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicExch(err, kErrWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_cluster(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, int* err) {
    return wait_phase(bar, parity, abort_flag, err, WAIT_LIMIT_NS, true);
}

// Tile t in grouped order: groups of `group` tile-rows, column by column within a group.
__host__ __device__ __forceinline__ void tile_coords_g(int t, int tiles_m, int tiles_n, int group,
                                                      int& tm, int& tn) {
    const int group_tiles = group * tiles_n;
    const int g = t / group_tiles;
    const int first = g * group;
    const int rows = min(group, tiles_m - first);
    const int r = t - g * group_tiles;
    tm = first + r % rows;
    tn = r / rows;
}

__host__ __device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm,
                                                    int& tn) {
    tile_coords_g(t, tiles_m, tiles_n, GROUP_M, tm, tn);
}

// Work decomposition over 256 x 256 output tiles in grouped order, one unit per CTA
// pair at a time. The first `full_tiles` tiles are computed whole and written to C.
// Each of the remaining `split_tiles` tiles is computed in `splits` parts over
// consecutive ranges of `kps` reduction blocks; a part writes its FP32 partial tile to
// block row `slot` of the partial plane (256 columns, splits * split_tiles * 256 rows),
// and a second kernel adds the parts in a fixed order. Alternatively (never both) the
// tiles after `full_tiles` are recut into `pieces` narrower units of whole reductions,
// at most one per pair: piece p covers rows [256 tm, +256) and columns [32 c, 32 (c + n))
// of C, with tm, c and n packed into piece[p] (bits 0-7, 8-15 and 16-20). Each CTA of a
// pair loads piece_box rows of B^T per plane for a piece (half the widest piece's columns;
// a narrower piece's MMAs read only the first n / 2 of them).
constexpr int MAX_PIECES = 128;
struct Work {
    int tiles_m, tiles_n, kblocks;
    int full_tiles, split_tiles, splits, kps;
    int pieces, piece_box;
    uint32_t piece[MAX_PIECES];
};

__host__ __device__ __forceinline__ uint32_t pack_piece(int tm, int col32, int width32) {
    return uint32_t(tm) | (uint32_t(col32) << 8) | (uint32_t(width32) << 16);
}

__host__ __device__ __forceinline__ int work_units(const Work& w) {
    return w.full_tiles + w.split_tiles * w.splits + w.pieces;
}

// Unit u: rows [256 tm, +256), columns [n0, n0 + nw), reduction blocks [kb0, kb1), and
// slot (-1: the unit writes C).
__host__ __device__ __forceinline__ void unit_coords(const Work& w, int u, int& tm, int& n0,
                                                     int& nw, int& kb0, int& kb1, int& slot) {
    int t, tn;
    if (u < w.full_tiles) {
        t = u;
        kb0 = 0;
        kb1 = w.kblocks;
        slot = -1;
    } else if (w.pieces > 0) {
        const uint32_t p = w.piece[u - w.full_tiles];
        tm = int(p & 0xffu);
        n0 = int((p >> 8) & 0xffu) * 32;
        nw = int((p >> 16) & 0x1fu) * 32;
        kb0 = 0;
        kb1 = w.kblocks;
        slot = -1;
        return;
    } else {
        // parts in part-major order: all pairs work in the same reduction range at a time
        const int v = u - w.full_tiles;
        const int part = v / w.split_tiles;
        const int r = v - part * w.split_tiles;
        t = w.full_tiles + r;
        kb0 = part * w.kps;
        kb1 = kb0 + w.kps < w.kblocks ? kb0 + w.kps : w.kblocks;
        slot = part * w.split_tiles + r;
    }
    tile_coords(t, w.tiles_m, w.tiles_n, tm, tn);
    n0 = tn * BN;
    nw = BN;
}

// Shared-memory layout and barriers (the same offsets in both CTAs of a pair).
// full[s]: leader only, completed by both CTAs' TMA bytes. empty[s]: both, arrived by
// the leader's multicast MMA commit. acc_full[b]: both, multicast commit. acc_empty[b]:
// leader only, arrived by every epilogue warp of both CTAs. drain: leader only.
struct Smem {
    uint32_t ring, bar0;
    uint32_t staging;    // shared address of the first staging block
    float* staging_ptr;  // the same, as a generic pointer
    uint32_t* tmem_slot;
    volatile int* abort_flag;
    __device__ uint32_t full(int s) const { return bar0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar0 + 8u * (MAX_STAGES + s); }
    __device__ uint32_t acc_full(int b) const { return bar0 + 8u * (2 * MAX_STAGES + b); }
    __device__ uint32_t acc_empty(int b) const { return bar0 + 8u * (2 * MAX_STAGES + 2 + b); }
    __device__ uint32_t drain() const { return bar0 + 8u * (2 * MAX_STAGES + 4); }
};

// Ring at the 1 KiB-aligned base, C staging right after it, barriers at a fixed offset.
template <class R>
__device__ __forceinline__ Smem carve_smem(uint8_t* smem_raw) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.ring = ptx::smem_u32(base);
    s.staging_ptr = reinterpret_cast<float*>(base + R::BYTES);
    s.staging = ptx::smem_u32(s.staging_ptr);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + RING_BYTES + STAGING_FIXED * STAGING_BYTES);
    s.bar0 = ptx::smem_u32(bars);
    s.tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
    return s;
}

// Barrier init (thread 0), tensor-map prefetch (warp 0) and the pair's TMEM allocation
// (warp 1 of each CTA); ends with a cluster barrier so that no CTA signals its peer's
// barriers before they exist. Returns the TMEM base address (the same in both CTAs).
template <class R>
__device__ __forceinline__ uint32_t setup(const Smem& sm, uint32_t acc_empty_count,
                                          const CUtensorMap* a_hi, const CUtensorMap* a_lo,
                                          const CUtensorMap* b_hi, const CUtensorMap* b_lo) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < R::STAGES; ++s) {
            ptx::mbar_init(sm.full(s), 1);
            ptx::mbar_init(sm.empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(sm.acc_full(b), 1);
            ptx::mbar_init(sm.acc_empty(b), acc_empty_count);
        }
        ptx::mbar_init(sm.drain(), 1);
        *sm.abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(a_hi);
        ptx::prefetch_tensormap(b_hi);
        if (R::PLANES == 2) {
            ptx::prefetch_tensormap(a_lo);
            ptx::prefetch_tensormap(b_lo);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_u32(sm.tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    // Launched with programmatic stream serialization right after the operand pre-pass:
    // everything above overlapped its tail; nothing below may touch memory it writes
    // before it has completed. The split-reduction kernel that may follow only waits.
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    return *sm.tmem_slot;
}

// Both CTAs leave the main loops, meet at a cluster barrier (so neither frees memory
// or TMEM its peer may still touch), then free the pair's TMEM together.
__device__ __forceinline__ void teardown(uint32_t tmem_base) {
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    if ((threadIdx.x >> 5) == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

__device__ __forceinline__ float rna_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// x truncated to TF32 (its 13 low mantissa bits cleared): the 3xTF32 high part.
__device__ __forceinline__ float trunc_tf32(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

// The 3xTF32 low part: x minus its high part (exact), rounded to TF32.
__device__ __forceinline__ float lo_tf32(float x) { return rna_tf32(x - trunc_tf32(x)); }

// ------------------------------------------------- A's split inside the GEMM kernel --
// With the fused split, A's rows are split into the hi/lo planes by warps of the GEMM
// kernel itself while earlier tiles are multiplied. Work is claimed from counters[0] in
// chunks of 1024 columns: first the rows the first round of tiles reads, chunk by chunk
// (chunk 0 of every such row, a few rows per claim, then chunk 1, ...), so that every
// pair can start on its first reduction blocks after a fraction of that split; then the
// remaining rows in ascending order, a whole row per claim. counters[1 + rb * MAX_SPLIT_CHUNKS + c] counts
// the finished rows of 256-row block rb in chunk c, and the TMA producer waits for a
// block's chunk to be complete before loading from it. A warp that has claimed work
// never waits on anything, so every claim is finished whatever the other CTAs are doing.
struct FusedSplit {
    const float* a;     // A (M x N, row-major); null: A was split before the launch
    float* a_hi;        // hi plane, row pitch N; null for 3xTF32 when A is its own hi
    float* a_lo;        // 3xTF32: the lo plane (row pitch N)
    int* counters;      // 1 + MAX_ROW_BLOCKS * MAX_SPLIT_CHUNKS ints, zero at launch
    int N;              // a multiple of 4, with A 16-byte aligned (the planes' pitch is N)
    int chunks;         // column chunks per row: ceil(N / 1024)
    int eager_rows;     // leading rows split chunk by chunk (the first round's rows)
};
constexpr int MAX_ROW_BLOCKS = 8192 / BM;
constexpr int FUSED_SPLIT_UNROLL = 8;  // 128-bit loads in flight per lane
constexpr int SPLIT_CHUNK4 = 32 * FUSED_SPLIT_UNROLL;         // float4s per claimed chunk
constexpr int MAX_SPLIT_CHUNKS = 8192 / (4 * SPLIT_CHUNK4);  // chunks of the longest row
constexpr int KB_PER_CHUNK = 4 * SPLIT_CHUNK4 / BK;          // reduction blocks per chunk
// rows per chunk-by-chunk claim: measured best at 4 for 3xTF32 and 2 for 1xTF32 (1, 2, 4
// tried; smaller claims start the MMAs sooner but stretch the split)
template <int PLANES>
__host__ __device__ constexpr int eager_rows_per_claim() { return PLANES == 1 ? 2 : 4; }
static_assert(4 * SPLIT_CHUNK4 % BK == 0 && MAX_SPLIT_CHUNKS <= 32 &&
                  BM % eager_rows_per_claim<1>() == 0 && BM % eager_rows_per_claim<2>() == 0,
              "chunks of whole reduction blocks, one publishing lane per chunk");

// The first chunk of the rows a fused GEMM's first round reads, prepared by the operand
// pre-pass (all SMs at DRAM speed, where the GEMM's splitting warps would take about 15 us
// before the first MMA): the pre-pass writes those planes and starts the GEMM's counters
// with the chunk's claims taken and its row counts complete.
struct PrepFirst {
    const float* a = nullptr;  // A (dense rows of n4 float4s, 16-byte aligned); null: none
    float* hi = nullptr;       // 1xTF32: the rounded plane; 3xTF32: the hi plane, or null
    float* lo = nullptr;       // 3xTF32: the lo plane
    int rows = 0;              // the first round's rows (whole 256-row blocks, or M)
    int c4 = 0;                // float4 columns of the chunk
    int n4 = 0;                // float4 columns of a row
    int blocks = 0;            // CTAs of the pre-pass that do it
    int M = 0;
    int claims = 0;            // the chunk's claims (rows per claim as in split_claimed)
};

__device__ __forceinline__ float4 rna_tf32_4(const float4& x) {
    return make_float4(rna_tf32(x.x), rna_tf32(x.y), rna_tf32(x.z), rna_tf32(x.w));
}

// One warp prepares chunk c of row r of A (float4 columns [c * SPLIT_CHUNK4, +SPLIT_CHUNK4)
// clipped to the row, one 128-bit load per lane and unrolled step): 1xTF32 (PLANES == 1)
// writes hi = rna(x); 3xTF32 (PLANES == 2) writes lo, and hi (x truncated) unless A
// itself is the hi operand (a_hi null). Rows are 16-byte aligned (N % 4 == 0); loads
// and plane stores are evict-first, so that the split traffic does not push the GEMM's
// operands out of L2.
template <int PLANES>
__device__ __forceinline__ void split_chunk(const FusedSplit& f, int r, int c, int lane) {
    constexpr int U = FUSED_SPLIT_UNROLL;
    const int n4 = f.N >> 2;
    const float4* src = reinterpret_cast<const float4*>(f.a) + size_t(r) * n4;
    float4* hi = f.a_hi ? reinterpret_cast<float4*>(f.a_hi) + size_t(r) * n4 : nullptr;
    float4* lo = PLANES == 2 ? reinterpret_cast<float4*>(f.a_lo) + size_t(r) * n4 : nullptr;
    const int c0 = c * SPLIT_CHUNK4 + lane;
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        x[u] = c0 + 32 * u < n4 ? __ldcs(src + c0 + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (c0 + 32 * u < n4) {
            const float4 v = x[u];
            if (PLANES == 1) {
                __stcs(hi + c0 + 32 * u, rna_tf32_4(v));
            } else {
                if (hi)
                    __stcs(hi + c0 + 32 * u, make_float4(trunc_tf32(v.x), trunc_tf32(v.y),
                                                         trunc_tf32(v.z), trunc_tf32(v.w)));
                __stcs(lo + c0 + 32 * u,
                       make_float4(lo_tf32(v.x), lo_tf32(v.y), lo_tf32(v.z), lo_tf32(v.w)));
            }
        }
    }
}

// The calling warp claims chunks (first) and rows (then) and splits them until the
// claims run out, or, with `eager_only`, until the chunk-by-chunk claims run out (a claim
// taken is always finished, also a whole row claimed past them). Each claim is published
// after its plane writes: they become visible, also to TMA, before lane c adds the row to
// chunk c's count.
template <int PLANES>
__device__ __forceinline__ void split_claimed(const FusedSplit& f, int M, bool eager_only) {
    const int lane = threadIdx.x & 31;
    constexpr int G = eager_rows_per_claim<PLANES>();
    const int E = f.eager_rows;
    const int groups = (E + G - 1) / G;  // eager claims per chunk
    const int eager_claims = groups * f.chunks;
    while (true) {
        int i = 0;
        if (lane == 0) i = atomicAdd(f.counters, 1);
        i = __shfl_sync(0xffffffffu, i, 0);
        int r0, r1, c_first, c_last;
        if (i < eager_claims) {
            // rows [G q, G q + G) of the eager rows, one chunk (never two row blocks)
            c_first = c_last = i / groups;
            r0 = (i - c_first * groups) * G;
            r1 = r0 + G < E ? r0 + G : E;
        } else {
            if (i - eager_claims >= M - E) return;
            r0 = E + (i - eager_claims);
            r1 = r0 + 1;
            c_first = 0;
            c_last = f.chunks - 1;
        }
        for (int r = r0; r < r1; ++r)
            for (int c = c_first; c <= c_last; ++c) split_chunk<PLANES>(f, r, c, lane);
        ptx::fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane >= c_first && lane <= c_last)
            ptx::red_release_gpu_add(f.counters + 1 + (r0 / BM) * MAX_SPLIT_CHUNKS + lane,
                                     r1 - r0);
        if (eager_only && i + 1 >= eager_claims) return;
    }
}

// Producer side: waits until chunk c of row block tm of A has been split (bounded like
// every wait).
__device__ __forceinline__ bool wait_rows(const FusedSplit& f, int tm, int c, int M,
                                          volatile int* abort_flag, int* err) {
    const int rows = M - tm * BM < BM ? M - tm * BM : BM;
    const int* done = f.counters + 1 + tm * MAX_SPLIT_CHUNKS + c;
    if (ptx::ld_acquire_gpu(done) < rows) {
        const unsigned long long t0 = global_ns();
        while (ptx::ld_acquire_gpu(done) < rows) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                atomicExch(err, kErrWaitTimeout);
                return false;
            }
        }
    }
    ptx::fence_proxy_async_global();  // the TMA loads that follow see the split rows
    return true;
}

// TMA producer (one thread per CTA): this CTA's halves of the A and B^T planes for every
// reduction block of every unit of the pair, one stage per block, each load
// signalling the leader's full barrier (which expects both CTAs' bytes). With a fused
// split (`fs` not null) it first waits for each chunk of a row block of A it reaches to
// be split, until one whole unit of that row block has been checked.
template <class R, bool F16 = false>
__device__ __forceinline__ void produce(const Smem& sm, uint32_t rank, const CUtensorMap* a_hi,
                                        const CUtensorMap* a_lo, const CUtensorMap* b_hi,
                                        const CUtensorMap* b_lo, const CUtensorMap* bp_hi,
                                        const CUtensorMap* bp_lo, const Work& w, int* err,
                                        const FusedSplit* fs = nullptr, int M = 0) {
    int s = 0;
    uint32_t ph = 0;
    const int units = work_units(w);
    const int pairs = gridDim.x >> 1;
    uint32_t ready = 0;  // row blocks of A known to be split in every chunk (bit tm)
    for (int u = blockIdx.x >> 1; u < units; u += pairs) {
        int tm, n0, nw, kb0, kb1, slot;
        unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
        const bool check = fs && !(ready >> tm & 1u);
        const int arow = tm * BM + int(rank) * HALF_M;
        // each CTA holds half of the unit's columns: a whole tile's 128 rows of B^T, or for
        // a recut piece one box of piece_box rows, of which its MMAs read the first nw / 2
        // (boxes of 16 rows, several per plane, were measured 4-23 % slower)
        const int brow = n0 + int(rank) * (nw >> 1);
        const bool piece = nw != BN;
        const CUtensorMap* bh = piece ? bp_hi : b_hi;
        const CUtensorMap* bl = piece ? bp_lo : b_lo;
        const uint32_t stage_tx =  // both CTAs' bytes
            2u * uint32_t(R::PLANES) * uint32_t((HALF_M + (piece ? w.piece_box : HALF_N)) * BK * 4);
        for (int kb = kb0; kb < kb1; ++kb) {
            if (check && (kb == kb0 || kb % KB_PER_CHUNK == 0) &&
                !wait_rows(*fs, tm, kb / KB_PER_CHUNK, M, sm.abort_flag, err))
                return;
            if (!wait_cluster(sm.empty(s), ph ^ 1u, sm.abort_flag, err)) return;
            const uint32_t full_leader = ptx::mapa_shared(sm.full(s), 0);
            const uint32_t st = sm.ring + uint32_t(s) * R::STAGE_BYTES;
            if (rank == 0) ptx::mbar_arrive_expect_tx(sm.full(s), stage_tx);
            const int kx = kb * BK_ELEMS<F16>;  // first reduction element of the block
            ptx::tma_load_2d_pair(st + R::a_off(0), a_hi, full_leader, kx, arow);
            if (R::PLANES == 2) ptx::tma_load_2d_pair(st + R::a_off(1), a_lo, full_leader, kx, arow);
            ptx::tma_load_2d_pair(st + R::b_off(0), bh, full_leader, kx, brow);
            if (R::PLANES == 2) ptx::tma_load_2d_pair(st + R::b_off(1), bl, full_leader, kx, brow);
            if (++s == R::STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (check && kb0 == 0 && kb1 == w.kblocks) ready |= 1u << tm;  // every chunk seen
    }
}

// A (128 rows per CTA) or B^T (128 rows per CTA) plane block in a stage: rows of 128
// bytes along the reduction, 8-row groups 1024 bytes apart (SBO); the k-th 32-byte slice
// starts 32 k bytes into each row.
__device__ __forceinline__ uint64_t plane_desc(uint32_t plane, int k) {
    return smem_desc_sw128(plane + uint32_t(k) * 32u, 16, 1024);
}

// The pair MMAs of one stage into d_tmem (both CTAs' TMEM), 256 x N with N from the
// instruction descriptor; the first of them overwrites when `fresh`. With two planes,
// each 32-byte slice k (8 floats or 16 halves) issues A_lo.B_hi, A_hi.B_lo and A_hi.B_hi
// (small terms first).
template <class R, bool F16 = false>
__device__ __forceinline__ void mma_stage(uint32_t st, uint32_t d_tmem, bool fresh,
                                          uint32_t idesc) {
    using ptx::Collect;
    const uint32_t a_hi = st + R::a_off(0), b_hi = st + R::b_off(0);
    // four 32-byte slices per 128-byte row: K = 8 floats or 16 halves each
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t first = (fresh && k == 0) ? 0u : 1u;
        if (R::PLANES == 2) {
            const uint32_t a_lo = st + R::a_off(1), b_lo = st + R::b_off(1);
            ptx::mma_pair<F16>(d_tmem, plane_desc(a_lo, k), plane_desc(b_hi, k), idesc, first);
            ptx::mma_pair<F16, Collect::fill>(d_tmem, plane_desc(a_hi, k), plane_desc(b_lo, k),
                                              idesc, 1u);
            ptx::mma_pair<F16, Collect::lastuse>(d_tmem, plane_desc(a_hi, k),
                                                 plane_desc(b_hi, k), idesc, 1u);
        } else {
            ptx::mma_pair<F16>(d_tmem, plane_desc(a_hi, k), plane_desc(b_hi, k), idesc, first);
        }
    }
}

// After an abort: let MMAs already issued finish before TMEM is released.
__device__ __forceinline__ void drain_mmas(const Smem& sm) {
    ptx::mma_commit_pair(sm.drain(), 0x1);
    const unsigned long long t0 = global_ns();
    while (!ptx::mbar_try_wait(sm.drain(), 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
    }
}

// Writes a 32-row x 32-column block of C for which TMA cannot be used (rows of C not
// 16-byte aligned): lane l supplies row r0 + l, columns c0 .. c0 + 31, from
// v[OFF .. OFF + 31]. The warp transposes the block through its first staging block (the
// same swizzled layout as the TMA path, conflict-free both ways), then writes it one row
// at a time, 32 consecutive floats per store instruction. Elements outside C are skipped.
template <int OFF, int NBUF, int NV>
__device__ __forceinline__ void store_block_direct(const Smem& sm, int ew, const float (&v)[NV],
                                                   int r0, int c0, int M, int K, float* C) {
    const int lane = threadIdx.x & 31;
    if (r0 >= M || c0 >= K) return;  // warp-uniform
    float* buf = sm.staging_ptr + ew * NBUF * (STAGING_BYTES / 4);
    if (lane == 0) ptx::bulk_wait_read0();  // no TMA store of this warp still reads it
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(buf + lane * 32 + ((c ^ (lane & 7)) * 4)) =
            make_float4(v[OFF + 4 * c], v[OFF + 4 * c + 1], v[OFF + 4 * c + 2], v[OFF + 4 * c + 3]);
    __syncwarp();
    const int col = c0 + lane;
    const int rows = M - r0 < 32 ? M - r0 : 32;
    if (col < K) {
        float* dst = C + size_t(r0) * K + col;
        const int chunk = lane >> 2, within = lane & 3;
#pragma unroll 8
        for (int rr = 0; rr < rows; ++rr)
            dst[size_t(rr) * K] = buf[rr * 32 + (((chunk ^ (rr & 7)) << 2) | within)];
    }
    __syncwarp();  // every lane has read the block before it is rewritten
}

// Writes a 32-row x 32-column block of C through one of epilogue warp `ew`'s NBUF
// staging blocks (used in turn; `nb` is the warp's rotation counter) and one TMA tensor
// store: lane l supplies row r0 + l, columns c0 .. c0 + 31, from v[OFF .. OFF + 31].
// Before a block is rewritten, the store that last used it must have read it: at most
// NBUF - 1 of the warp's stores may still be reading. The block is written in the
// 128-byte swizzled layout the tensor map expects (16-byte chunk c of row l at chunk
// c ^ (l % 8)), which also keeps the warp's shared-memory stores free of bank conflicts.
// Rows and columns outside C are clipped by the tensor map.
template <int OFF, int NBUF, int NV>
__device__ __forceinline__ void store_block_tma(const Smem& sm, int ew, int& nb,
                                                const CUtensorMap* tmC, const float (&v)[NV],
                                                int r0, int c0, int M, int K) {
    const int lane = threadIdx.x & 31;
    if (r0 >= M || c0 >= K) return;  // warp-uniform
    const int j = ew * NBUF + nb;
    nb = nb + 1 == NBUF ? 0 : nb + 1;
    float* buf = sm.staging_ptr + j * (STAGING_BYTES / 4);
    if (lane == 0) ptx::bulk_wait_read<NBUF - 1>();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4*>(buf + lane * 32 + ((c ^ (lane & 7)) * 4)) =
            make_float4(v[OFF + 4 * c], v[OFF + 4 * c + 1], v[OFF + 4 * c + 2], v[OFF + 4 * c + 3]);
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_2d(tmC, sm.staging + uint32_t(j * STAGING_BYTES), c0, r0);
        ptx::bulk_commit();
    }
}

// ------------------------------------------------ kernel 1: one accumulator per tile --
// 1xTF32. Launched in clusters of two CTAs; CTA rank r of a pair owns rows
// [tm * 256 + 128 r, +128) of each of the pair's tiles. FUSED: A's rounding is done by
// this kernel (warps 6-9 throughout, the epilogue warps at the start).
template <bool FUSED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED ? THREADS_TILE_FUSED : THREADS_TILE, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA_hi,
                   const __grid_constant__ CUtensorMap tmA_lo,
                   const __grid_constant__ CUtensorMap tmB_hi,
                   const __grid_constant__ CUtensorMap tmB_lo,
                   const __grid_constant__ CUtensorMap tmBp_hi,
                   const __grid_constant__ CUtensorMap tmBp_lo,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmP, float* __restrict__ C, int M, int K,
                   Work w, int tma_store, int* err, const FusedSplit fs) {
    using R = Ring1;
    constexpr int NBUF = R::STAGING_BLOCKS / EPI_WARPS_TILE;
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve_smem<R>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int units = work_units(w);
    const int pairs = gridDim.x >> 1;
    const uint32_t tmem_base =
        setup<R>(sm, 2 * EPI_WARPS_TILE, &tmA_hi, &tmA_lo, &tmB_hi, &tmB_lo);

    if (warp == 0) {
        if (lane == 0)
            produce<R>(sm, rank, &tmA_hi, &tmA_lo, &tmB_hi, &tmB_lo, &tmBp_hi, &tmBp_lo, w, err,
                       FUSED ? &fs : nullptr, M);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool issued = false;
            for (int u = blockIdx.x >> 1; u < units; u += pairs, ++it) {
                int tm, n0, nw, kb0, kb1, slot;
                unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
                const uint32_t idesc = idesc_tf32(BM, nw);
                const int b = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!wait_cluster(sm.acc_empty(b), aph ^ 1u, sm.abort_flag, err)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + uint32_t(b * BN);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_cluster(sm.full(s), ph, sm.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (!issued) clock_mark(0);
                    mma_stage<R>(sm.ring + uint32_t(s) * R::STAGE_BYTES, d_tmem, kb == kb0, idesc);
                    issued = true;
                    ptx::mma_commit_pair(sm.empty(s), PAIR_MASK);
                    if (++s == R::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(sm.acc_full(b), PAIR_MASK);
            }
            if (*sm.abort_flag && issued) drain_mmas(sm);
        }
    } else if (FUSED && warp >= 2 + EPI_WARPS_TILE) {
        split_claimed<1>(fs, M, false);
    } else {
        // epilogue: warps 2-5, TMEM -> registers -> C (or this split's partial plane);
        // with the fused split they first help round the rows the first tiles need
        if (FUSED) split_claimed<1>(fs, M, true);
        const int q = warp & 3;  // this warp may read TMEM lanes [32 q, 32 q + 32)
        int it = 0;
        int nb = 0;
        for (int u = blockIdx.x >> 1; u < units; u += pairs, ++it) {
            int tm, n0, nw, kb0, kb1, slot;
            unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
            const int row0 = tm * BM + int(rank) * HALF_M + q * 32;
            // split parts go to their block row of the partial plane
            const int prow0 = slot * BM + int(rank) * HALF_M + q * 32;
            const int prows = w.splits * w.split_tiles * BM;
            const int b = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!wait_cluster(sm.acc_full(b), aph, sm.abort_flag, err)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(b * BN);
#pragma unroll 1
            for (int c = 0; c < nw; c += 32) {
                uint32_t r0[16], r1[16];
                __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
                ptx::tmem_ld_16(taddr + c, r0);
                ptx::tmem_ld_16(taddr + c + 16, r1);
                float v[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v[i] = __uint_as_float(r0[i]);
                    v[16 + i] = __uint_as_float(r1[i]);
                }
                if (slot >= 0) {
                    store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmP, v, prow0, c, prows, BN);
                } else if (tma_store) {
                    store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmC, v, row0, n0 + c, M, K);
                } else {
                    store_block_direct<0, NBUF>(sm, warp - 2, v, row0, n0 + c, M, K, C);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(sm.acc_empty(b), 0));
        }
        if (lane == 0) ptx::bulk_wait0();
        if (warp == 2 && lane == 0) clock_mark(1);  // CTA 0's stores are done
    }
    teardown(tmem_base);
}

// ------------------------------- kernel 2: 3 products with segmented accumulation ----
// Segment g (counted over all units of the pair) accumulates SEG_KB reduction blocks
// (SEG_KB stages, 12 * SEG_KB pair MMAs) into TMEM buffer g % 2, starting from zero; the epilogue warps
// of both CTAs add it into per-thread FP32 registers and free the buffer. FUSED: A's
// split is done by this kernel (warps 10-11 throughout, the epilogue warps at the start).
// F16: the planes hold FP16 hi/lo pieces of A and B scaled by powers of two (A's row m by
// 2^ea[m], B's columns k in block k / 128 by 2^eb[k / 128]); kind::f16 MMAs, and the
// epilogue multiplies each sum by 2^-(ea[m] + eb[k / 128]) before storing it (exact,
// barring underflow).
template <bool FUSED, bool F16 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED ? THREADS_SEG_FUSED : THREADS_SEG, 1)
    tc_gemm_seg_kernel(const __grid_constant__ CUtensorMap tmA_hi,
                       const __grid_constant__ CUtensorMap tmA_lo,
                       const __grid_constant__ CUtensorMap tmB_hi,
                       const __grid_constant__ CUtensorMap tmB_lo,
                       const __grid_constant__ CUtensorMap tmBp_hi,
                       const __grid_constant__ CUtensorMap tmBp_lo,
                       const __grid_constant__ CUtensorMap tmC,
                       const __grid_constant__ CUtensorMap tmP, float* __restrict__ C, int M,
                       int K, Work w, int tma_store, int* err, const FusedSplit fs,
                       const int* __restrict__ ea, const int* __restrict__ eb) {
    using R = Ring3;
    constexpr int NBUF = R::STAGING_BLOCKS / EPI_WARPS_SEG;
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve_smem<R>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int units = work_units(w);
    const int pairs = gridDim.x >> 1;
    const uint32_t tmem_base =
        setup<R>(sm, 2 * EPI_WARPS_SEG, &tmA_hi, &tmA_lo, &tmB_hi, &tmB_lo);

    if (warp == 0) {
        if (lane == 0)
            produce<R, F16>(sm, rank, &tmA_hi, &tmA_lo, &tmB_hi, &tmB_lo, &tmBp_hi, &tmBp_lo, w,
                            err, FUSED ? &fs : nullptr, M);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int g = 0;  // segment counter across units
            bool issued = false;
            bool ok = true;
            for (int u = blockIdx.x >> 1; ok && u < units; u += pairs) {
                int tm, n0, nw, kb0, kb1, slot;
                unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
                const uint32_t idesc = F16 ? idesc_f16(BM, nw) : idesc_tf32(BM, nw);
                const int segs = (kb1 - kb0 + SEG_KB - 1) / SEG_KB;
                for (int sg = 0; sg < segs; ++sg, ++g) {
                    const int b = g & 1;
                    const uint32_t aph = (g >> 1) & 1;
                    if (!wait_cluster(sm.acc_empty(b), aph ^ 1u, sm.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + uint32_t(b * BN);
                    const int s0 = kb0 + sg * SEG_KB;
                    const int s1 = min(kb1, s0 + SEG_KB);
                    for (int kb = s0; kb < s1; ++kb) {
                        if (!wait_cluster(sm.full(s), ph, sm.abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if (!issued) clock_mark(0);
                        mma_stage<R, F16>(sm.ring + uint32_t(s) * R::STAGE_BYTES, d_tmem, kb == s0,
                                          idesc);
                        issued = true;
                        ptx::mma_commit_pair(sm.empty(s), PAIR_MASK);
                        if (++s == R::STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair(sm.acc_full(b), PAIR_MASK);
                }
            }
            if (*sm.abort_flag && issued) drain_mmas(sm);
        }
    } else if (FUSED && warp >= 2 + EPI_WARPS_SEG) {
        split_claimed<2>(fs, M, false);
    } else {
        // epilogue: warps 2-9. Warp w reads TMEM lanes [32 (w % 4), +32) and columns
        // [128 h, 128 h + 128) with h = (w - 2) / 4; each thread owns one row's 128
        // running sums. With the fused split they first help split the rows the first
        // tiles need.
        if (FUSED) split_claimed<2>(fs, M, true);
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        float acc[128];
        int g = 0;
        int nb = 0;
        bool ok = true;
        for (int u = blockIdx.x >> 1; ok && u < units; u += pairs) {
            int tm, n0, nw, kb0, kb1, slot;
            unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
            const int segs = (kb1 - kb0 + SEG_KB - 1) / SEG_KB;
            // segment g's accumulator: wait until it is complete, return its TMEM address
            auto seg_wait = [&](int gg, uint32_t& taddr) {
                const int b = gg & 1;
                if (!wait_cluster(sm.acc_full(b), uint32_t(gg >> 1) & 1u, sm.abort_flag, err))
                    return false;
                ptx::tc_fence_after();
                taddr = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(b * BN + h * 128);
                return true;
            };
            // hand segment g's TMEM buffer back to the MMA warp
            auto seg_free = [&](int gg) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive_cluster(ptx::mapa_shared(sm.acc_empty(gg & 1), 0));
            };
            uint32_t taddr;
            if (!seg_wait(g, taddr)) {
                ok = false;
                break;
            }
            // the tile's first segment initialises the sums: two wide loads, no adds
#pragma unroll
            for (int c = 0; c < 128; c += 64) {
                uint32_t r[64];
                __syncwarp();
                ptx::tmem_ld_64(taddr + c, r);
#pragma unroll
                for (int i = 0; i < 64; ++i) acc[c + i] = __uint_as_float(r[i]);
            }
            seg_free(g++);
            for (int sg = 1; sg < segs; ++sg, ++g) {
                if (!seg_wait(g, taddr)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 128; c += 16) {
                    uint32_t r[16];
                    __syncwarp();
                    ptx::tmem_ld_16(taddr + c, r);
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[c + i] += __uint_as_float(r[i]);
                }
                seg_free(g);
            }
            if (!ok) break;
            const int row0 = tm * BM + int(rank) * HALF_M + q * 32;
            if constexpr (F16) {
                // undo the operands' power-of-two scales: row row0 + lane, columns
                // n0 + 128 h + c (exact unless the result underflows)
                const int r = row0 + lane;
                const int er = r < M ? __ldg(ea + r) : 0;
                // this thread's 128 columns meet at most two of B's 128-column scale blocks
                const int cb = n0 + h * 128;
                const int nb = (K + F16_COL_BLOCK - 1) / F16_COL_BLOCK;
                const int b0 = min(cb / F16_COL_BLOCK, nb - 1);
                const int b1 = min((cb + 127) / F16_COL_BLOCK, nb - 1);
                const int split_col = (b0 + 1) * F16_COL_BLOCK - cb;  // columns in block b0
                const int e0 = er + __ldg(eb + b0), e1 = er + __ldg(eb + b1);
                if (e0 >= -126 && e0 <= 126 && e1 >= -126 && e1 <= 126) {
                    // 2^-e as normal floats (the common case): one multiply per sum
                    const float f0 = __int_as_float((127 - e0) << 23);
                    const float f1 = __int_as_float((127 - e1) << 23);
#pragma unroll
                    for (int c = 0; c < 128; ++c) acc[c] *= c < split_col ? f0 : f1;
                } else {
#pragma unroll
                    for (int c = 0; c < 128; ++c) acc[c] = ldexpf(acc[c], -(c < split_col ? e0 : e1));
                }
            }
            if (slot >= 0) {
                // a split part: its block row of the partial plane, local columns
                const int r0 = slot * BM + int(rank) * HALF_M + q * 32, c0 = h * 128;
                const int rl = w.splits * w.split_tiles * BM;
                store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmP, acc, r0, c0, rl, BN);
                store_block_tma<32, NBUF>(sm, warp - 2, nb, &tmP, acc, r0, c0 + 32, rl, BN);
                store_block_tma<64, NBUF>(sm, warp - 2, nb, &tmP, acc, r0, c0 + 64, rl, BN);
                store_block_tma<96, NBUF>(sm, warp - 2, nb, &tmP, acc, r0, c0 + 96, rl, BN);
            } else {
                // blocks of 32 columns inside the unit (a narrow unit has fewer; warp h
                // may have none, its sums of unused TMEM columns are dropped)
                const int c0 = n0 + h * 128, left = nw - h * 128;
                if (tma_store) {
                    if (left > 0) store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmC, acc, row0, c0, M, K);
                    if (left > 32) store_block_tma<32, NBUF>(sm, warp - 2, nb, &tmC, acc, row0, c0 + 32, M, K);
                    if (left > 64) store_block_tma<64, NBUF>(sm, warp - 2, nb, &tmC, acc, row0, c0 + 64, M, K);
                    if (left > 96) store_block_tma<96, NBUF>(sm, warp - 2, nb, &tmC, acc, row0, c0 + 96, M, K);
                } else {
                    if (left > 0) store_block_direct<0, NBUF>(sm, warp - 2, acc, row0, c0, M, K, C);
                    if (left > 32) store_block_direct<32, NBUF>(sm, warp - 2, acc, row0, c0 + 32, M, K, C);
                    if (left > 64) store_block_direct<64, NBUF>(sm, warp - 2, acc, row0, c0 + 64, M, K, C);
                    if (left > 96) store_block_direct<96, NBUF>(sm, warp - 2, acc, row0, c0 + 96, M, K, C);
                }
            }
        }
        if (lane == 0) ptx::bulk_wait0();
        if (warp == 2 && lane == 0) clock_mark(1);  // CTA 0's stores are done
    }
    teardown(tmem_base);
}

// ------------------------------------------ kernel 3: 1xTF32 on 256 x 512 pair tiles --
// On 256 x 256 tiles a 1xTF32 stage (32 KiB per CTA) feeds only 4 MMAs. On 256 x 512
// tiles a stage of 48 KiB per CTA (A 128 rows, B^T 256 rows) feeds 8: the TMA fills per
// MMA drop by a quarter, and so does the L2 traffic per flop. The accumulator takes all
// 512 TMEM columns, so the MMAs of a unit wait until the epilogue has drained the last.
// The schedule takes whole 256 x 512 tiles in grouped order; the tiles of a partly filled
// last round are split in two along the reduction when their parts fit in one round, and
// wide_reduce_kernel adds the two partial tiles. At 8192^3 it measured 4 % faster than the
// 256 x 256 kernel; where its rounds quantize worse it is not used (use_wide).
constexpr int BN_W = 2 * BN;  // columns of a wide tile
struct WideWork {
    int tiles_m, wtiles_n, kblocks, K;
    int group;       // tile-rows per group of the grouped order
    int wide_units;  // units [0, wide_units): whole wide tiles in grouped order
    int tail_tiles;  // the next wide tiles, each computed in two parts, over reduction
                     // blocks [0, kps) and [kps, kblocks), listed part by part
    int kps;
};
__host__ __device__ __forceinline__ int wide_units_total(const WideWork& w) {
    return w.wide_units + 2 * w.tail_tiles;
}
// Unit u: rows [256 tm, +256), columns [n0, n0 + nw) with nw 512, or 256 for a tile whose
// right half lies past K; reduction blocks [kb0, kb1); slot (-1: the unit writes C, else
// its block row of the partial plane, part * tail_tiles + tail tile).
__host__ __device__ __forceinline__ void wide_unit(const WideWork& w, int u, int& tm, int& n0,
                                                   int& nw, int& kb0, int& kb1, int& slot) {
    int t = u;
    kb0 = 0;
    kb1 = w.kblocks;
    slot = -1;
    if (u >= w.wide_units) {
        const int v = u - w.wide_units;
        const int part = v / w.tail_tiles, r = v - part * w.tail_tiles;
        t = w.wide_units + r;
        kb0 = part == 0 ? 0 : w.kps;
        kb1 = part == 0 ? w.kps : w.kblocks;
        slot = v;
    }
    int tn;
    tile_coords_g(t, w.tiles_m, w.wtiles_n, w.group, tm, tn);
    n0 = tn * BN_W;
    nw = n0 + BN >= w.K ? BN : BN_W;
}

// Ring of the wide kernel: per stage this CTA's 128 x 32 block of the A plane, then two
// 128 x 32 blocks of the B^T plane (rows n0 + 256 h + 128 rank, h = 0, 1).
constexpr int W_STAGES = 4;
constexpr int W_STAGE_BYTES = A_PLANE_BYTES + 2 * B_PLANE_BYTES;  // 48 KiB
constexpr int W_EPI_WARPS = 8;  // two per TMEM lane quarter, each 256 of the 512 columns
constexpr int W_EPI_COLS = BN_W * 4 / W_EPI_WARPS;  // columns drained by one epilogue warp
constexpr int THREADS_WIDE = 64 + 32 * W_EPI_WARPS;  // TMA warp, MMA warp, epilogue
// with A's rounding fused: six more warps that round A's rows (a round of wide tiles
// consumes rows about twice as fast as a round of 256 x 256 tiles)
constexpr int THREADS_WIDE_FUSED = THREADS_WIDE + 192;
static_assert(W_STAGES * W_STAGE_BYTES == RING_BYTES, "the wide ring fills the ring budget");
static_assert(W_STAGES <= MAX_STAGES, "barrier slots");
struct RingW {
    static constexpr int PLANES = 1;
    static constexpr int STAGES = W_STAGES;
    static constexpr int BYTES = RING_BYTES;
};

template <bool FUSED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(FUSED ? THREADS_WIDE_FUSED : THREADS_WIDE, 1)
    tc_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                        float* __restrict__ C, int M, int K, WideWork w, int tma_store, int* err,
                        const FusedSplit fs) {
    constexpr int NBUF = STAGING_FIXED / W_EPI_WARPS;
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve_smem<RingW>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int units = wide_units_total(w);
    const int pairs = gridDim.x >> 1;
    const uint32_t tmem_base = setup<RingW>(sm, 2 * W_EPI_WARPS, &tmA, &tmA, &tmB, &tmB);

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer: A block and one or two B^T blocks per reduction block
            int s = 0;
            uint32_t ph = 0;
            uint32_t ready = 0;  // row blocks of A known to be split in every chunk
            for (int u = blockIdx.x >> 1; u < units; u += pairs) {
                int tm, n0, nw, kb0, kb1, slot;
                wide_unit(w, u, tm, n0, nw, kb0, kb1, slot);
                const bool check = FUSED && !(ready >> tm & 1u);
                const int arow = tm * BM + int(rank) * HALF_M;
                const uint32_t stage_tx =  // both CTAs' bytes
                    2u * uint32_t(A_PLANE_BYTES + (nw == BN_W ? 2 : 1) * B_PLANE_BYTES);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (check && (kb == kb0 || kb % KB_PER_CHUNK == 0) &&
                        !wait_rows(fs, tm, kb / KB_PER_CHUNK, M, sm.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    if (!wait_cluster(sm.empty(s), ph ^ 1u, sm.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = ptx::mapa_shared(sm.full(s), 0);
                    const uint32_t st = sm.ring + uint32_t(s) * W_STAGE_BYTES;
                    if (rank == 0) ptx::mbar_arrive_expect_tx(sm.full(s), stage_tx);
                    const int kx = kb * BK;
                    ptx::tma_load_2d_pair(st, &tmA, full_leader, kx, arow);
                    ptx::tma_load_2d_pair(st + A_PLANE_BYTES, &tmB, full_leader, kx,
                                          n0 + int(rank) * HALF_N);
                    if (nw == BN_W)
                        ptx::tma_load_2d_pair(st + A_PLANE_BYTES + B_PLANE_BYTES, &tmB, full_leader,
                                              kx, n0 + BN + int(rank) * HALF_N);
                    if (++s == W_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                if (check && kb0 == 0 && kb1 == w.kblocks) ready |= 1u << tm;  // every chunk seen
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool issued = false;
            constexpr uint32_t idesc = idesc_tf32(BM, BN);
            for (int u = blockIdx.x >> 1; u < units; u += pairs) {
                int tm, n0, nw, kb0, kb1, slot;
                wide_unit(w, u, tm, n0, nw, kb0, kb1, slot);
                // the accumulator of the previous unit must have been drained
                if (!wait_cluster(sm.acc_empty(0), (uint32_t(it) & 1u) ^ 1u, sm.abort_flag, err)) break;
                ptx::tc_fence_after();
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_cluster(sm.full(s), ph, sm.abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (!issued) clock_mark(0);
                    const uint32_t st = sm.ring + uint32_t(s) * W_STAGE_BYTES;
                    const uint32_t b0 = st + A_PLANE_BYTES, b1 = b0 + B_PLANE_BYTES;
                    // the four slices into columns [0, 256), then (wide units) into
                    // [256, 512): consecutive MMAs into one accumulator (measured faster
                    // than alternating them to reuse A from the collector buffer)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ptx::mma_pair<false>(tmem_base, plane_desc(st, k), plane_desc(b0, k), idesc,
                                             (kb == kb0 && k == 0) ? 0u : 1u);
                    if (nw == BN_W) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            ptx::mma_pair<false>(tmem_base + uint32_t(BN), plane_desc(st, k),
                                                 plane_desc(b1, k), idesc,
                                                 (kb == kb0 && k == 0) ? 0u : 1u);
                    }
                    issued = true;
                    ptx::mma_commit_pair(sm.empty(s), PAIR_MASK);
                    if (++s == W_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit_pair(sm.acc_full(0), PAIR_MASK);
                ++it;
            }
            if (*sm.abort_flag && issued) drain_mmas(sm);
        }
    } else if (FUSED && warp >= 2 + W_EPI_WARPS) {
        split_claimed<1>(fs, M, false);
    } else {
        // epilogue: warp w drains TMEM lanes [32 (w % 4), +32), columns [W_EPI_COLS h,
        // +W_EPI_COLS) with h = (w - 2) / 4, in 32-column blocks through TMA stores. With
        // the fused split they first help round the rows the first tiles need.
        if (FUSED) split_claimed<1>(fs, M, true);
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        int it = 0;
        int nb = 0;
        for (int u = blockIdx.x >> 1; u < units; u += pairs) {
            int tm, n0, nw, kb0, kb1, slot;
            wide_unit(w, u, tm, n0, nw, kb0, kb1, slot);
            if (!wait_cluster(sm.acc_full(0), uint32_t(it) & 1u, sm.abort_flag, err)) break;
            ptx::tc_fence_after();
            const int row0 = tm * BM + int(rank) * HALF_M + q * 32;
            const uint32_t taddr = tmem_base + (uint32_t(q * 32) << 16);
            const int c_end = (h + 1) * W_EPI_COLS < nw ? (h + 1) * W_EPI_COLS : nw;
            {
#pragma unroll 1
                for (int c = h * W_EPI_COLS; c < c_end; c += 32) {
                    uint32_t r0[16], r1[16];
                    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
                    ptx::tmem_ld_16(taddr + c, r0);
                    ptx::tmem_ld_16(taddr + c + 16, r1);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[i] = __uint_as_float(r0[i]);
                        v[16 + i] = __uint_as_float(r1[i]);
                    }
                    const int col = n0 + c;
                    if (slot >= 0)  // a tail part: its block row of the partial plane
                        store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmP, v,
                                                 slot * BM + int(rank) * HALF_M + q * 32, c,
                                                 2 * w.tail_tiles * BM, BN_W);
                    else if (tma_store)
                        store_block_tma<0, NBUF>(sm, warp - 2, nb, &tmC, v, row0, col, M, K);
                    else
                        store_block_direct<0, NBUF>(sm, warp - 2, v, row0, col, M, K, C);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(sm.acc_empty(0), 0));
            ++it;
        }
        if (lane == 0) ptx::bulk_wait0();
        if (warp == 2 && lane == 0) clock_mark(1);  // CTA 0's stores are done
    }
    teardown(tmem_base);
}

// ---------------------------------------------------------------- wait self-test ---
// One CTA waits, through wait_phase, on an mbarrier that nothing ever completes. The
// wait must give up after limit_ns, raise the device error word and return, leaving
// the context usable: the path every GEMM role takes if a hand-off never arrives.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int* err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        wait_phase(ptx::smem_u32(&bar), 0, &abort_flag, err, limit_ns);
    __syncthreads();
}

// ---------------------------------------------------------------- rate probe -------
// The pair MMA rate with nothing else in the way: each CTA fills its 128 rows of one A
// block and one B^T block in shared memory once (128-byte rows, 32 floats or 64 halves;
// values k/8 with |k| <= 8, exact in TF32 and FP16 and not all alike, so the datapath
// switches as on real data), then the leader issues `iters` reduction blocks of four
// M=256 N=256 pair MMAs (K=8 for kind::tf32, K=16 for kind::f16) into one TMEM
// accumulator and a single multicast commit. The descriptors and the instruction forms
// are the GEMM kernels'. Every wait is bounded as in the GEMM.
template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    mma_probe_kernel(int iters, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* blocks = reinterpret_cast<float*>(base);  // A half, then B^T half
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + A_PLANE_BYTES + B_PLANE_BYTES);
    uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = ptx::cluster_ctarank();
    constexpr int FLOATS = (A_PLANE_BYTES + B_PLANE_BYTES) / 4;
    for (int i = threadIdx.x; i < FLOATS; i += blockDim.x) {
        uint32_t h = uint32_t(i) * 2654435761u + rank * 40503u;
        h ^= h >> 15;
        const float v = float(int(h % 17u) - 8) * 0.125f;
        if constexpr (F16) {
            const __half2 two = __floats2half2_rn(v, -0.5f * v);  // both exact in FP16
            blocks[i] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&two));
        } else {
            blocks[i] = v;
        }
    }
    ptx::fence_proxy_async_smem();
    const uint32_t done = ptx::smem_u32(bars), drain = ptx::smem_u32(bars + 1);
    if (threadIdx.x == 0) {
        ptx::mbar_init(done, 1);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc_pair(ptx::smem_u32(slot), BN);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t a_blk = ptx::smem_u32(blocks), b_blk = a_blk + A_PLANE_BYTES;
    if (rank == 0 && threadIdx.x == 0) {
        constexpr uint32_t idesc = F16 ? idesc_f16(BM, BN) : idesc_tf32(BM, BN);
        clock_mark(0);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                ptx::mma_pair<F16>(tmem, plane_desc(a_blk, k), plane_desc(b_blk, k), idesc,
                                   (it | k) ? 1u : 0u);
        }
        ptx::mma_commit_pair(done, PAIR_MASK);
    }
    const bool finished = threadIdx.x == 0 ? wait_phase(done, 0, abort_flag, err) : true;
    if (threadIdx.x == 0 && rank == 0 && finished) clock_mark(1);
    if (threadIdx.x == 0 && !finished && rank == 0) {
        // let MMAs already issued finish before TMEM is released
        ptx::mma_commit_pair(drain, 0x1);
        const unsigned long long t0 = global_ns();
        while (!ptx::mbar_try_wait(drain, 0) && global_ns() - t0 < WAIT_LIMIT_NS) {
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    if (warp == 0) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, BN);
    }
}

// ---------------------------------------------------------------- operand split ----

// One launch prepares both operands (and zeroes `nzero` ints at `zero`, if not null: the
// GEMM's counters). Blocks [0, a_blocks) prepare A (M x N, dense rows)
// into plane(s) with row pitch lda; the remaining blocks each transpose one PREP_BT x PREP_BT tile
// of B (N x K) into B^T planes (K x N, row pitch ldbt). 1xTF32 (PLANES == 1) writes the
// rounded values; 3xTF32 writes hi = x truncated and lo, and for A only lo when a_hi is
// null (the GEMM then loads A itself as its hi plane).
template <int PLANES>
__global__ void __launch_bounds__(256)
    tf32_prep_kernel(const float* __restrict__ a, int M, int N, int lda, float* a_hi, float* a_lo,
                     int vec_a, int a_blocks, const float* __restrict__ b, int K, int ldbt,
                     float* bt_hi, float* bt_lo, int b_tiles_k, int* zero, int nzero,
                     const PrepFirst first) {
    ptx::griddep_launch_dependents();  // the GEMM may start its set-up beside this grid
    if (zero && blockIdx.x == 0) {
        // the fused GEMM's counters: zero, except for the first chunk done here
        for (int i = int(threadIdx.x); i < nzero; i += int(blockDim.x)) {
            int v = 0;
            if (first.a) {
                const int rb = (i - 1) / MAX_SPLIT_CHUNKS, c = (i - 1) % MAX_SPLIT_CHUNKS;
                if (i == 0)
                    v = first.claims;
                else if (c == 0 && rb < MAX_ROW_BLOCKS && rb * BM < first.rows)
                    v = first.M - rb * BM < BM ? first.M - rb * BM : BM;
            }
            zero[i] = v;
        }
    }
    if (int(blockIdx.x) >= a_blocks && int(blockIdx.x) < a_blocks + first.blocks) {
        // the first chunk of the first round's rows (PLANES == 1: rounded; 2: lo, and hi
        // unless A is its own hi plane), PREP_A_UNROLL 128-bit loads in flight per thread
        const size_t total = size_t(first.rows) * first.c4;
        const size_t stride = size_t(first.blocks) * blockDim.x;
        const float4* src = reinterpret_cast<const float4*>(first.a);
        for (size_t i = size_t(int(blockIdx.x) - a_blocks) * blockDim.x + threadIdx.x; i < total;
             i += stride * PREP_A_UNROLL) {
            float4 xs[PREP_A_UNROLL];
            size_t at[PREP_A_UNROLL];
#pragma unroll
            for (int u = 0; u < PREP_A_UNROLL; ++u) {
                const size_t j = i + size_t(u) * stride;
                const size_t r = j / first.c4, c = j - r * first.c4;
                at[u] = r * first.n4 + c;
                xs[u] = j < total ? __ldcs(src + at[u]) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < PREP_A_UNROLL; ++u) {
                if (i + size_t(u) * stride >= total) break;
                const float4 x = xs[u];
                if (PLANES == 2) {
                    if (first.hi)
                        __stcs(reinterpret_cast<float4*>(first.hi) + at[u],
                               make_float4(trunc_tf32(x.x), trunc_tf32(x.y), trunc_tf32(x.z),
                                           trunc_tf32(x.w)));
                    __stcs(reinterpret_cast<float4*>(first.lo) + at[u],
                           make_float4(lo_tf32(x.x), lo_tf32(x.y), lo_tf32(x.z), lo_tf32(x.w)));
                } else {
                    __stcs(reinterpret_cast<float4*>(first.hi) + at[u], rna_tf32_4(x));
                }
            }
        }
        return;
    }
    if (int(blockIdx.x) < a_blocks) {
        const size_t total = size_t(M) * N;
        const size_t stride = size_t(a_blocks) * blockDim.x;
        size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
        if (vec_a) {
            // dense rows (lda == N, N % 4 == 0) and a 16-byte aligned source
            // PREP_A_UNROLL 128-bit loads in flight per thread before the dependent stores
            const size_t n4 = total / 4;
            for (; i < n4; i += stride * PREP_A_UNROLL) {
                float4 xs[PREP_A_UNROLL];
#pragma unroll
                for (int u = 0; u < PREP_A_UNROLL; ++u) {
                    const size_t j = i + size_t(u) * stride;
                    xs[u] = j < n4 ? __ldcs(reinterpret_cast<const float4*>(a) + j)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < PREP_A_UNROLL; ++u) {
                    const size_t j = i + size_t(u) * stride;
                    if (j >= n4) break;
                    const float4 x = xs[u];
                    if (PLANES == 2) {
                        if (a_hi)
                            __stcs(reinterpret_cast<float4*>(a_hi) + j,
                                   make_float4(trunc_tf32(x.x), trunc_tf32(x.y), trunc_tf32(x.z),
                                               trunc_tf32(x.w)));
                        __stcs(reinterpret_cast<float4*>(a_lo) + j,
                               make_float4(lo_tf32(x.x), lo_tf32(x.y), lo_tf32(x.z), lo_tf32(x.w)));
                    } else {
                        __stcs(reinterpret_cast<float4*>(a_hi) + j,
                               make_float4(rna_tf32(x.x), rna_tf32(x.y), rna_tf32(x.z),
                                           rna_tf32(x.w)));
                    }
                }
            }
        } else {
            // rows that are not 16-byte aligned: a warp per row, lanes along the row
            const int lane = threadIdx.x & 31;
            const int warps = a_blocks * int(blockDim.x >> 5);
            for (int r = int(blockIdx.x) * int(blockDim.x >> 5) + int(threadIdx.x >> 5); r < M;
                 r += warps) {
                const float* src = a + size_t(r) * N;
                float* hi = a_hi ? a_hi + size_t(r) * lda : nullptr;
                float* lo = PLANES == 2 ? a_lo + size_t(r) * lda : nullptr;
                // eight loads in flight per lane before the dependent stores
                constexpr int U = 8;
                for (int c0 = lane; c0 < N; c0 += 32 * U) {
                    float x[U];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        x[u] = c0 + 32 * u < N ? __ldcs(src + c0 + 32 * u) : 0.0f;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (c0 + 32 * u < N) {
                            if (hi) hi[c0 + 32 * u] = PLANES == 2 ? trunc_tf32(x[u]) : rna_tf32(x[u]);
                            if (PLANES == 2) lo[c0 + 32 * u] = lo_tf32(x[u]);
                        }
                    }
                }
            }
        }
        return;
    }
    // a BT x BT tile of B per block: each thread has BT * BT / 256 loads in flight
    __shared__ float tile[PREP_BT][PREP_BT + 1];
    constexpr int ROWS = 256 / PREP_BT;  // tile rows covered by one pass of the block
    // tiles in reverse order: the last ones written, still in L2 when the GEMM starts, are
    // the first reduction rows of the first output columns, which its first round reads
    // first (measured 0.2-0.3 % faster steps than the forward order)
    const int t = int(gridDim.x) - 1 - int(blockIdx.x);
    const int k0 = (t % b_tiles_k) * PREP_BT;
    const int n0 = (t / b_tiles_k) * PREP_BT;
    const int tx = threadIdx.x % PREP_BT, ty = threadIdx.x / PREP_BT;
#pragma unroll
    for (int i = 0; i < PREP_BT / ROWS; ++i) {
        const int n = n0 + ty + ROWS * i, k = k0 + tx;
        tile[ty + ROWS * i][tx] = (n < N && k < K) ? __ldcs(b + size_t(n) * K + k) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < PREP_BT / ROWS; ++i) {
        const int k = k0 + ty + ROWS * i, n = n0 + tx;
        if (k < K && n < N) {
            const float x = tile[tx][ty + ROWS * i];
            // (a truncated hi plane, not x itself: B operands whose low 13 bits are not
            // zero made the pair MMAs about 2 % slower, although the tensor core ignores
            // those bits; A's made no measurable difference)
            bt_hi[size_t(k) * ldbt + n] = PLANES == 2 ? trunc_tf32(x) : rna_tf32(x);
            if (PLANES == 2) bt_lo[size_t(k) * ldbt + n] = lo_tf32(x);
        }
    }
}

// ------------------------------------------ FP16 pieces with power-of-two scales ----
// For the FP16 three-product path each row m of A is multiplied by 2^ea[m] and each block
// of 128 columns of B by 2^eb[block], chosen so that the row's (block's) largest
// magnitude lands in [2^14, 2^15): FP16's normal range then holds the hi piece of every
// element within 2^28 of that largest one and the lo piece (x - hi, about 2^-11 of x) of
// every element within 2^17. (A scale per block rather than per column lets the GEMM's
// epilogue undo it with one or two factors per thread.) hi = x rounded to FP16 and lo = (x - hi) rounded to FP16 (x - hi is exact
// in FP32), 22 significant bits in all. The maxima leave out Inf and NaN elements
// (finite_mag), so one non-finite input cannot set the scale of its neighbours; it still
// propagates through its own products (its lo piece is Inf - Inf = NaN). A zero maximum
// (no finite non-zero element) gives scale 1.
__device__ __forceinline__ uint32_t finite_mag(uint32_t bits) {
    const uint32_t mag = bits & 0x7fffffffu;
    return mag >= 0x7f800000u ? 0u : mag;  // exponent field all ones: Inf or NaN
}

__device__ __forceinline__ int scale_exponent(uint32_t max_bits) {
    const float m = __uint_as_float(max_bits);
    if (!(m > 0.0f) || !isfinite(m)) return 0;  // zero, NaN or Inf
    return 14 - ilogbf(m);
}

__device__ __forceinline__ void split_f16(float x, int e, __half& hi, __half& lo) {
    const float xs = ldexpf(x, e);  // exact: a power-of-two scale
    hi = __float2half_rn(xs);
    lo = __float2half_rn(xs - __half2float(hi));
}

// Pass 1: the largest finite magnitude of each 128-column block of B (a CTA per 32-row
// strip of 256 columns; each warp merges its 32 columns with atomicMax), as the bit
// patterns of |x|, whose unsigned order is their numeric order. bmax is zero at launch.
__global__ void __launch_bounds__(256)
    f16_colmax_kernel(const float* __restrict__ b, int N, int K, int b_cols, uint32_t* bmax) {
    const int k = (int(blockIdx.x) % b_cols) * 256 + int(threadIdx.x);
    const int n0 = (int(blockIdx.x) / b_cols) * 32;
    uint32_t m = 0;
    if (k < K)
        for (int n = n0; n < n0 + 32 && n < N; ++n)
            m = max(m, finite_mag(__float_as_uint(__ldcs(b + size_t(n) * K + k))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int k_warp = k - (int(threadIdx.x) & 31);  // the warp's first column
    if ((threadIdx.x & 31) == 0 && k_warp < K) atomicMax(bmax + k_warp / F16_COL_BLOCK, m);
}

// Pass 2: A's scaled hi/lo planes (a warp per row; row pitch lda halves) and B^T's
// (64 x 64 transpose tiles, as in the TF32 pre-pass; row pitch ldbt halves), and the
// exponents ea, eb that the GEMM's epilogue undoes. A row's maximum is found by the same
// warp, in a first read of the row whose lines the second read then finds in L2.
__global__ void __launch_bounds__(256)
    f16_split_kernel(const float* __restrict__ a, int M, int N, int lda, __half* a_hi,
                     __half* a_lo, int a_blocks, int vec_a, int* ea,
                     const float* __restrict__ b, int K, int ldbt, __half* bt_hi,
                     __half* bt_lo, int b_tiles_k, const uint32_t* __restrict__ bmax, int* eb) {
    ptx::griddep_launch_dependents();  // the GEMM may start its set-up beside this grid
    const int lane = threadIdx.x & 31;
    if (int(blockIdx.x) < a_blocks) {
        const int warps = a_blocks * 8;
        for (int r = int(blockIdx.x) * 8 + int(threadIdx.x >> 5); r < M; r += warps) {
            const float* row = a + size_t(r) * N;
            uint32_t m = 0;
            if (vec_a) {
                const int n4 = N >> 2;
                for (int c = lane; c < n4; c += 32) {
                    const float4 x = reinterpret_cast<const float4*>(row)[c];
                    m = max(max(m, finite_mag(__float_as_uint(x.x))),
                            max(max(finite_mag(__float_as_uint(x.y)),
                                    finite_mag(__float_as_uint(x.z))),
                                finite_mag(__float_as_uint(x.w))));
                }
            } else {
                for (int c = lane; c < N; c += 32) m = max(m, finite_mag(__float_as_uint(row[c])));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            const int e = scale_exponent(m);
            if (lane == 0) ea[r] = e;
            __half* hrow = a_hi + size_t(r) * lda;
            __half* lrow = a_lo + size_t(r) * lda;
            if (vec_a) {
                // 16-byte aligned rows (N % 4 == 0): four 128-bit loads in flight per lane,
                // four halves (8 bytes) stored per plane and load
                constexpr int U = 4;
                const int n4 = N >> 2;
                for (int c0 = lane; c0 < n4; c0 += 32 * U) {
                    float4 x[U];
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        x[u] = c0 + 32 * u < n4 ? __ldcs(reinterpret_cast<const float4*>(row) + c0 + 32 * u)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + 32 * u;
                        if (c >= n4) break;
                        __half h[4], l[4];
                        split_f16(x[u].x, e, h[0], l[0]);
                        split_f16(x[u].y, e, h[1], l[1]);
                        split_f16(x[u].z, e, h[2], l[2]);
                        split_f16(x[u].w, e, h[3], l[3]);
                        *reinterpret_cast<uint2*>(hrow + 4 * c) = *reinterpret_cast<const uint2*>(h);
                        *reinterpret_cast<uint2*>(lrow + 4 * c) = *reinterpret_cast<const uint2*>(l);
                    }
                }
            } else {
                for (int c = lane; c < N; c += 32) {
                    __half h, l;
                    split_f16(__ldcs(row + c), e, h, l);
                    hrow[c] = h;
                    lrow[c] = l;
                }
            }
        }
        return;
    }
    __shared__ float tile[PREP_BT][PREP_BT + 1];
    constexpr int ROWS = 256 / PREP_BT;
    const int t = int(gridDim.x) - 1 - int(blockIdx.x);  // reverse order, as in tf32_prep
    const int k0 = (t % b_tiles_k) * PREP_BT;
    const int n0 = (t / b_tiles_k) * PREP_BT;
    const int tx = threadIdx.x % PREP_BT, ty = threadIdx.x / PREP_BT;
#pragma unroll
    for (int i = 0; i < PREP_BT / ROWS; ++i) {
        const int n = n0 + ty + ROWS * i, k = k0 + tx;
        tile[ty + ROWS * i][tx] = (n < N && k < K) ? __ldcs(b + size_t(n) * K + k) : 0.f;
    }
    __syncthreads();
    // B^T rows k: 32 threads per row, two consecutive n each (one 4-byte store per plane)
    const int px = threadIdx.x & 31, py = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < PREP_BT / 8; ++i) {
        const int kk = py + 8 * i, k = k0 + kk, n = n0 + 2 * px;
        if (k < K && n < N) {
            const int e = scale_exponent(bmax[k / F16_COL_BLOCK]);
            if (n == 0 && k % F16_COL_BLOCK == 0) eb[k / F16_COL_BLOCK] = e;
            __half h[2], l[2];
            split_f16(tile[2 * px][kk], e, h[0], l[0]);
            split_f16(tile[2 * px + 1][kk], e, h[1], l[1]);  // zero past N: padding
            *reinterpret_cast<uint32_t*>(bt_hi + size_t(k) * ldbt + n) = *reinterpret_cast<const uint32_t*>(h);
            *reinterpret_cast<uint32_t*>(bt_lo + size_t(k) * ldbt + n) = *reinterpret_cast<const uint32_t*>(l);
        }
    }
}

// ---------------------------------------------------------------- host side ----------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return EncodeTiledFn(nullptr);
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Row-major float32 plane (rows x cols, row pitch ld floats) with a box of
// box_cols x box_rows, 128-byte swizzle, zero fill outside rows x cols.
bool encode_plane(CUtensorMap* map, const float* base, int rows, int cols, int ld, int box_cols,
                  int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
    const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major FP16 plane (rows x cols, row pitch ld halves, a multiple of 8) with boxes of
// 64 x box_rows (128-byte rows, swizzled like the FP32 planes), zero fill outside.
bool encode_plane16(CUtensorMap* map, const __half* base, int rows, int cols, int ld,
                    int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
    const cuuint32_t box[2] = {64u, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pad8(int n) { return (n + 7) / 8 * 8; }
size_t round_halves(size_t n) { return (n + 127) / 128 * 128; }  // 256-byte plane starts

size_t round_floats(size_t n) { return (n + 63) / 64 * 64; }  // 256-byte plane starts
int pad4(int n) { return (n + 3) / 4 * 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Fixed-order sum of the split parts: for each of the `split_tiles` tiles (tile index
// full_tiles + r in grouped order), C = sum over part = 0 .. splits-1 of its block row
// part * split_tiles + r of the partial plane (256 columns per row).
__global__ void __launch_bounds__(256)
    split_reduce_kernel(const float* __restrict__ P, Work w, int M, int K, float* __restrict__ C) {
    ptx::griddep_wait();  // the GEMM's partial tiles are complete
    const size_t per_tile = size_t(BM) * BN;
    const size_t total = size_t(w.split_tiles) * per_tile;
    const size_t part_stride = size_t(w.split_tiles) * per_tile;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const int r = int(i / per_tile);
        const int e = int(i - size_t(r) * per_tile);
        const int lr = e / BN, lc = e - lr * BN;
        int tm, tn;
        tile_coords(w.full_tiles + r, w.tiles_m, w.tiles_n, tm, tn);
        const int m = tm * BM + lr, k = tn * BN + lc;
        if (m >= M || k >= K) continue;
        const float* p = P + i;
        float s = 0.f;
        for (int part = 0; part < w.splits; ++part) s += __ldcs(p + part * part_stride);
        C[size_t(m) * K + k] = s;
    }
}

int kblocks_of(int N) { return (N + BK - 1) / BK; }

// Recuts the tiles of a partly filled last round (all tiles when there is one round)
// into at most `pairs` pieces as narrow as possible, so that pairs without a tile in
// that round share its columns: in each 256-row block the last round's tiles form one
// run of columns up to the right edge of C, which is cut into pieces of equal width
// (multiples of 32). Every piece takes the whole reduction, so each element of C is
// summed exactly as in a full tile. Used when the widest piece's modelled time is at
// most 0.93 of a full tile's (3xTF32 only).
// Modelled cycles of one reduction block (32 wide) per CTA of the 3xTF32 kernel for a
// unit of nw columns: the larger of the MMA time (12 pair MMAs M=256, K=8 of 135 cycles
// at N = 256, proportional to N) and the shared-memory time (TMA fills of the four
// operand planes, nw / 2 rows of B^T, plus the MMAs' operand reads, at about 100 bytes
// per cycle; with full-height B boxes this reproduced the full tile's and a 96-column
// piece's measured times). A's share does not shrink with nw, so narrow pieces are bound
// by shared memory.
double block_cycles(int nw) {
    const double mma = 12.0 * 135.0 * nw / BN;
    const double bytes = 12.0 * (HALF_M + nw / 2) * UMMA_K * 4.0 + 2.0 * (HALF_M + nw / 2) * BK * 4.0;
    return mma > bytes / 100.0 ? mma : bytes / 100.0;
}

bool recut_last_round(Work& w, int K, int pairs) {
    const int tiles = w.tiles_m * w.tiles_n;
    const int rem = tiles % pairs;
    if (rem == 0 || pairs > MAX_PIECES) return false;
    int lo[8192 / BM], hi[8192 / BM], count[8192 / BM];
    if (w.tiles_m > 8192 / BM) return false;
    for (int r = 0; r < w.tiles_m; ++r) {
        lo[r] = w.tiles_n;
        hi[r] = -1;
        count[r] = 0;
    }
    for (int t = tiles - rem; t < tiles; ++t) {
        int tm, tn;
        tile_coords(t, w.tiles_m, w.tiles_n, tm, tn);
        lo[tm] = tn < lo[tm] ? tn : lo[tm];
        hi[tm] = tn > hi[tm] ? tn : hi[tm];
        ++count[tm];
    }
    int len[8192 / BM];  // columns of each row block's run
    for (int r = 0; r < w.tiles_m; ++r) {
        if (count[r] == 0) {
            len[r] = 0;
            continue;
        }
        if (count[r] != hi[r] - lo[r] + 1) return false;  // not one run
        const int end = (hi[r] + 1) * BN < K ? (hi[r] + 1) * BN : K;
        len[r] = end - lo[r] * BN;
    }
    int width = 0;
    for (int wd = 32; wd <= BN - 32 && width == 0; wd += 32) {
        int n = 0;
        for (int r = 0; r < w.tiles_m; ++r) n += (len[r] + wd - 1) / wd;
        if (n <= pairs) width = wd;
    }
    // worth it only if the recut round is clearly shorter than a round of full tiles (the
    // model is optimistic for wide pieces: 224 columns, rated 0.94, measured no faster)
    if (width == 0 || block_cycles(width) > 0.93 * block_cycles(BN)) return false;
    int p = 0;
    for (int r = 0; r < w.tiles_m; ++r) {
        if (len[r] == 0) continue;
        const int units32 = (len[r] + 31) / 32;
        const int n = (len[r] + width - 1) / width;
        const int q = units32 / n, extra = units32 % n;
        int col32 = lo[r] * (BN / 32);
        for (int i = 0; i < n; ++i) {
            const int wd32 = q + (i < extra ? 1 : 0);
            w.piece[p++] = pack_piece(r, col32, wd32);
            col32 += wd32;
        }
    }
    w.full_tiles = tiles - rem;
    w.pieces = p;
    w.piece_box = width / 2;
    return true;
}

// Schedule for a shape on `sm_count` SMs (sm_count / 2 CTA pairs, `passes` products per
// term). When the tiles are too few to keep the pairs busy, every tile is split along the
// reduction. A partly filled last round is split along the reduction, recut into narrower
// pieces, or left as is, whichever the cost model below rates fastest. (With the split
// parts listed tile by tile, so that pairs worked in different reduction ranges at once,
// a split of 8192 x 6144 x 4096's 56 trailing tiles did not shorten the GEMM.)
Work make_schedule(int M, int N, int K, int sm_count, int passes) {
    Work w;
    w.tiles_m = (M + BM - 1) / BM;
    w.tiles_n = (K + BN - 1) / BN;
    w.kblocks = kblocks_of(N);
    const int tiles = w.tiles_m * w.tiles_n;
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    w.full_tiles = tiles;
    w.split_tiles = 0;
    w.splits = 1;
    w.kps = w.kblocks;
    w.pieces = 0;
    w.piece_box = 0;
    const size_t part_bytes = size_t(BM) * BN * sizeof(float);
    const size_t max_plane = size_t(256) << 20;
    if (tiles * 4 < pairs * 3) {
        // too few tiles for the pairs: split every tile (at least 4 blocks per part)
        int splits = (pairs + tiles - 1) / tiles;
        if (splits > w.kblocks / 4) splits = w.kblocks / 4;
        if (splits > 32) splits = 32;
        while (splits > 1 && size_t(splits) * tiles * part_bytes > max_plane) --splits;
        if (splits > 1) {
            w.full_tiles = 0;
            w.split_tiles = tiles;
            w.splits = splits;
        }
    } else if (tiles * 4 >= pairs * 3 && tiles % pairs != 0) {
        // a partly filled last round (or a single round), modelled in rounds of whole
        // tiles: as is (1); recut into narrower pieces (3xTF32); or with its tiles split
        // along the reduction into `sp` parts, taken part by part by all pairs, plus the
        // partial planes' round trip through HBM and the reducing launch (at an effective
        // 4.8 TB/s, fitted to the measured gains at 4096^3 and 8192 x 6144 x 4096). A
        // recut whose pieces are at least 160 columns wide is taken whenever it applies
        // (at 8192 x 8192 x 1024 it beat a 4-part split by 3.6 %); narrower pieces are
        // costed by the model, which they exceed by about 0.07 (measured at 96 columns).
        const int rem = tiles % pairs;
        Work wr = w;
        double recut_cost = 2.0;
        if (passes == 3 && recut_last_round(wr, K, pairs))
            recut_cost = 2 * wr.piece_box >= 160
                             ? 0.0
                             : block_cycles(2 * wr.piece_box) / block_cycles(BN) + 0.07;
        const double t_round = w.kblocks * (passes == 3 ? 0.79e-6 : 0.27e-6);  // seconds
        int best = 1;
        double best_cost = 1.0;
        for (int sp = 2; tiles > pairs && sp <= 16 && sp <= w.kblocks / 4; ++sp) {
            const double rounds = double((rem * sp + pairs - 1) / pairs) / sp;
            const double extra =
                (double(rem) * (2 * sp + 1) * double(part_bytes) / 4.8e12 + 5.0e-6) / t_round;
            if (rounds + extra < best_cost - 1e-9 && size_t(sp) * rem * part_bytes <= max_plane) {
                best_cost = rounds + extra;
                best = sp;
            }
        }
        // (a split rated above 0.95 measured even: 8192 x 6144 x 4096, 4 parts, 0.97)
        if (best > 1 && best_cost < 0.95 && best_cost < recut_cost) {
            w.full_tiles = tiles - rem;
            w.split_tiles = rem;
            w.splits = best;
        } else if (recut_cost < 1.0) {
            w = wr;
        }
    }
    if (w.split_tiles > 0) {
        w.kps = (w.kblocks + w.splits - 1) / w.splits;
        w.splits = (w.kblocks + w.kps - 1) / w.kps;  // no empty part
    }
    return w;
}

// PASSES == 1: tile-accumulator kernel; PASSES == 3: segmented-accumulation kernel.
// Split parts write FP32 partial tiles to `partials` (block rows of 256 x 256) and
// split_reduce_kernel finishes those tiles.
// The 1xTF32 schedule on 256 x 512 tiles: whole tiles in grouped order; a partly filled
// last round whose tiles, in two parts each, fit in one round is split along the
// reduction (a wide_reduce_kernel launch adds the parts). (Computing those tiles as
// 256 x 256 halves instead ran at 0.74 of the tensor rate, against about 1.0 for wide
// units.)
// A group holds at least the tile-rows that one round covers, so that the first round
// reads few rows of A (which the GEMM can then round itself) and each round reads every
// row of A and column of B^T it needs once.
WideWork make_wide_schedule(int M, int N, int K, int sm_count) {
    WideWork w;
    w.tiles_m = (M + BM - 1) / BM;
    w.wtiles_n = (K + BN_W - 1) / BN_W;
    w.kblocks = kblocks_of(N);
    w.K = K;
    const int tiles = w.tiles_m * w.wtiles_n;
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int round_rows = (pairs + w.wtiles_n - 1) / w.wtiles_n;
    w.group = round_rows > GROUP_M ? round_rows : GROUP_M;
    const int rem = tiles % pairs;
    w.wide_units = tiles;
    w.tail_tiles = 0;
    w.kps = w.kblocks;
    if (rem != 0 && 2 * rem <= pairs && w.kblocks >= 8) {
        w.wide_units = tiles - rem;
        w.tail_tiles = rem;
        w.kps = w.kblocks / 2;
    }
    return w;
}

size_t wide_partial_bytes(const WideWork& w) {
    return size_t(2) * w.tail_tiles * BM * BN_W * sizeof(float);
}

// Whether a 1xTF32 product runs on 256 x 512 tiles: a reduction long enough that draining
// the single accumulator after each tile (a few microseconds) is small against the tile's
// MMAs, and fewer rounds than on 256 x 256 tiles, counted in 256 x 256 tile times: a wide
// tile takes WIDE_TILE_TIME of them (measured at 8192^3: 3.4 % faster than 256 x 256
// tiles with split last rounds), a split tail one; 256 x 256 tiles take whole rounds, or
// fill them, with 0.1 of a round's overhead, where their schedule splits or recuts a
// partly filled last round.
constexpr double WIDE_TILE_TIME = 1.86;
Work make_schedule(int M, int N, int K, int sm_count, int passes);
bool use_wide(int M, int N, int K, int sm_count) {
    if (N < 2048) return false;
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int tiles_m = (M + BM - 1) / BM;
    const int wtiles = tiles_m * ((K + BN_W - 1) / BN_W);
    if (wtiles < 2 * pairs) return false;
    const int rem = wtiles % pairs;
    const double wide = (wtiles / pairs) * WIDE_TILE_TIME +
                        (rem == 0 ? 0.0 : 2 * rem <= pairs ? 1.0 : WIDE_TILE_TIME);
    const Work n = make_schedule(M, N, K, sm_count, 1);
    const int tiles = n.tiles_m * n.tiles_n;
    const double narrow = n.split_tiles > 0 || n.pieces > 0 ? double(tiles) / pairs + 0.1
                                                           : double((tiles + pairs - 1) / pairs);
    return wide < 0.97 * narrow;
}

int first_round_rows_wide(const WideWork& w, int M, int pairs) {
    const int units = wide_units_total(w);
    int max_tm = 0;
    for (int u = 0; u < units && u < pairs; ++u) {
        int tm, n0, nw, kb0, kb1, slot;
        wide_unit(w, u, tm, n0, nw, kb0, kb1, slot);
        if (tm > max_tm) max_tm = tm;
    }
    return (max_tm + 1) * BM < M ? (max_tm + 1) * BM : M;
}

// Launches `kernel` with programmatic stream serialization: when the kernel before it in
// the stream signals (griddepcontrol.launch_dependents), this one may start and do its
// set-up while that one drains; it waits for it (griddepcontrol.wait) before touching
// memory. After any other stream operation it is an ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                              size_t smem, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Rows of A that the first round of units reads (the epilogue warps of a fused launch
// help split these before their first tile).
int first_round_rows(const Work& w, int M, int pairs) {
    const int units = work_units(w);
    const int first = units < pairs ? units : pairs;
    int max_tm = 0;
    for (int u = 0; u < first; ++u) {
        int tm, n0, nw, kb0, kb1, slot;
        unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
        if (tm > max_tm) max_tm = tm;
    }
    return (max_tm + 1) * BM < M ? (max_tm + 1) * BM : M;
}

template <int PASSES, bool F16 = false>
cudaError_t launch_gemm(const CUtensorMap& ah, const CUtensorMap& al, const CUtensorMap& bh,
                        const CUtensorMap& bl, const CUtensorMap& bph, const CUtensorMap& bpl,
                        float* C, int M, int N, int K, const Work& w,
                        float* partials, int sm_count, cudaStream_t stream,
                        const KernelTimer& timer, int* err, FusedSplit fs,
                        const int* ea = nullptr, const int* eb = nullptr) {
    static_assert(PASSES == 1 || PASSES == 3, "one or three products per term");
    static_assert(!F16 || PASSES == 3, "FP16 pieces come in three products");
    const bool fused = fs.a != nullptr;
    if (F16 && (fused || !ea || !eb)) return cudaErrorInvalidValue;
    cudaError_t e = F16        ? set_smem_limit_once<tc_gemm_seg_kernel<false, true>>(SMEM_BYTES)
                    : PASSES == 1 ? (fused ? set_smem_limit_once<tc_gemm_kernel<true>>(SMEM_BYTES)
                                           : set_smem_limit_once<tc_gemm_kernel<false>>(SMEM_BYTES))
                    : fused     ? set_smem_limit_once<tc_gemm_seg_kernel<true>>(SMEM_BYTES)
                                : set_smem_limit_once<tc_gemm_seg_kernel<false>>(SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int units = work_units(w);
    const int max_pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int grid = 2 * (units < max_pairs ? units : max_pairs);  // clusters of two CTAs
    const int vec_store = (K % 4 == 0 && aligned16(C)) ? 1 : 0;
    alignas(64) CUtensorMap tc, tp;
    int tma_store = 0;
    // TMA-store epilogue when C is a TMA-legal tensor (16-byte aligned rows)
    if (w.full_tiles > 0 && vec_store && encode_plane(&tc, C, M, K, K, 32, 32))
        tma_store = 1;
    else
        tc = ah;  // unused
    if (w.split_tiles > 0) {
        if (!encode_plane(&tp, partials, w.splits * w.split_tiles * BM, BN, BN, 32, 32))
            return cudaErrorInvalidValue;
    } else {
        tp = ah;  // unused
    }
    if (fused) fs.eager_rows = first_round_rows(w, M, max_pairs);
    timer.before();
    const int* ep = ea;
    const int* bp = eb;
    if (F16)
        e = launch_overlapped(tc_gemm_seg_kernel<false, true>, grid, THREADS_SEG, SMEM_BYTES,
                              stream, ah, al, bh, bl, bph, bpl, tc, tp, C, M, K, w, tma_store, err,
                              fs, ep, bp);
    else if (PASSES == 1 && fused)
        e = launch_overlapped(tc_gemm_kernel<true>, grid, THREADS_TILE_FUSED, SMEM_BYTES, stream,
                              ah, al, bh, bl, bph, bpl, tc, tp, C, M, K, w, tma_store, err, fs);
    else if (PASSES == 1)
        e = launch_overlapped(tc_gemm_kernel<false>, grid, THREADS_TILE, SMEM_BYTES, stream, ah,
                              al, bh, bl, bph, bpl, tc, tp, C, M, K, w, tma_store, err, fs);
    else if (fused)
        e = launch_overlapped(tc_gemm_seg_kernel<true>, grid, THREADS_SEG_FUSED, SMEM_BYTES,
                              stream, ah, al, bh, bl, bph, bpl, tc, tp, C, M, K, w, tma_store, err,
                              fs, ep, bp);
    else
        e = launch_overlapped(tc_gemm_seg_kernel<false>, grid, THREADS_SEG, SMEM_BYTES, stream,
                              ah, al, bh, bl, bph, bpl, tc, tp, C, M, K, w, tma_store, err, fs, ep,
                              bp);
    timer.after();
    count_launch();
    if (e != cudaSuccess || w.split_tiles == 0) return e;
    const size_t total = size_t(w.split_tiles) * BM * BN;
    size_t blocks = (total + 255) / 256;
    const size_t cap = size_t(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    const float* pp = partials;
    e = launch_overlapped(split_reduce_kernel, unsigned(blocks), 256, 0, stream, pp, w, M, K, C);
    count_launch();
    return e;
}

// The wide schedule's tail: C = P_0 + P_1 over each tail tile (its two parts' block rows of
// the partial plane, 512 columns each), in that order. Four consecutive columns per thread.
__global__ void __launch_bounds__(256)
    wide_reduce_kernel(const float* __restrict__ P, WideWork w, int M, int K, float* __restrict__ C) {
    ptx::griddep_wait();  // the GEMM's partial tiles are complete
    const size_t per_tile4 = size_t(BM) * BN_W / 4;
    const size_t total = size_t(w.tail_tiles) * per_tile4;
    const float4* P4 = reinterpret_cast<const float4*>(P);
    const bool vec = (K & 3) == 0 && (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const int r = int(i / per_tile4);
        const int e = int(i - size_t(r) * per_tile4) * 4;
        const int lr = e / BN_W, lc = e - lr * BN_W;
        int tm, tn;
        tile_coords_g(w.wide_units + r, w.tiles_m, w.wtiles_n, w.group, tm, tn);
        const int m = tm * BM + lr, k = tn * BN_W + lc;
        if (m >= M || k >= K) continue;
        const float4 a = __ldcs(P4 + i), b = __ldcs(P4 + i + total);
        const float4 v = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
        float* dst = C + size_t(m) * K + k;
        if (vec) {
            *reinterpret_cast<float4*>(dst) = v;  // K % 4 == 0: the 4 columns are inside
        } else {
            dst[0] = v.x;
            if (k + 1 < K) dst[1] = v.y;
            if (k + 2 < K) dst[2] = v.z;
            if (k + 3 < K) dst[3] = v.w;
        }
    }
}

cudaError_t launch_wide(const CUtensorMap& ah, const CUtensorMap& bh, float* C, int M, int N,
                        int K, float* partials, int sm_count, cudaStream_t stream,
                        const KernelTimer& timer, int* err, FusedSplit fs) {
    const bool fused = fs.a != nullptr;
    cudaError_t e = fused ? set_smem_limit_once<tc_gemm_wide_kernel<true>>(SMEM_BYTES)
                          : set_smem_limit_once<tc_gemm_wide_kernel<false>>(SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const WideWork w = make_wide_schedule(M, N, K, sm_count);
    const int units = wide_units_total(w);
    const int max_pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int grid = 2 * (units < max_pairs ? units : max_pairs);
    alignas(64) CUtensorMap tc, tp;
    const int tma_store = (K % 4 == 0 && aligned16(C) && encode_plane(&tc, C, M, K, K, 32, 32)) ? 1 : 0;
    if (!tma_store) tc = ah;  // unused
    if (w.tail_tiles > 0) {
        if (!partials || !encode_plane(&tp, partials, 2 * w.tail_tiles * BM, BN_W, BN_W, 32, 32))
            return cudaErrorInvalidValue;
    } else {
        tp = ah;  // unused
    }
    if (fused) fs.eager_rows = first_round_rows_wide(w, M, max_pairs);
    timer.before();
    if (fused)
        e = launch_overlapped(tc_gemm_wide_kernel<true>, grid, THREADS_WIDE_FUSED, SMEM_BYTES,
                              stream, ah, bh, tc, tp, C, M, K, w, tma_store, err, fs);
    else
        e = launch_overlapped(tc_gemm_wide_kernel<false>, grid, THREADS_WIDE, SMEM_BYTES, stream,
                              ah, bh, tc, tp, C, M, K, w, tma_store, err, fs);
    timer.after();
    count_launch();
    if (e != cudaSuccess || w.tail_tiles == 0) return e;
    const size_t total4 = size_t(w.tail_tiles) * BM * BN_W / 4;
    size_t blocks = (total4 + 255) / 256;
    const size_t cap = size_t(sm_count > 0 ? sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    const float* pp = partials;
    e = launch_overlapped(wide_reduce_kernel, unsigned(blocks), 256, 0, stream, pp, w, M, K, C);
    count_launch();
    return e;
}

}  // namespace

cudaError_t launch_wait_selftest(long long limit_ns, int* err, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_ns, err);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_mma_probe(bool f16, int iters, int sm_count, int* err, cudaStream_t stream,
                             const KernelTimer& timer) {
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int smem = A_PLANE_BYTES + B_PLANE_BYTES + 1024 + 64;
    // load the kernel before the start event, so that a lazy module load is not timed
    cudaFuncAttributes attr;
    cudaError_t e = f16 ? cudaFuncGetAttributes(&attr, mma_probe_kernel<true>)
                        : cudaFuncGetAttributes(&attr, mma_probe_kernel<false>);
    if (e != cudaSuccess) return e;
    timer.before();
    if (f16)
        mma_probe_kernel<true><<<2 * pairs, 128, smem, stream>>>(iters, err);
    else
        mma_probe_kernel<false><<<2 * pairs, 128, smem, stream>>>(iters, err);
    e = cudaGetLastError();
    timer.after();
    count_launch();
    return e;
}

double mma_probe_flops(bool f16, int iters, int sm_count) {
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    return double(pairs) * iters * 4 * 2.0 * BM * BN * (f16 ? 16 : 8);
}

int tc_schedule_units(int M, int N, int K, int passes, int sm_count, int* out, int cap) {
    if (passes == 1 && use_wide(M, N, K, sm_count)) {
        const WideWork ww = make_wide_schedule(M, N, K, sm_count);
        int n = 0;
        for (int u = 0; u < wide_units_total(ww); ++u) {
            int tm, n0, nw, kb0, kb1, slot;
            wide_unit(ww, u, tm, n0, nw, kb0, kb1, slot);
            if (n < cap) {
                int* o = out + 6 * size_t(n);
                o[0] = tm * BM;
                o[1] = n0;
                o[2] = nw;
                o[3] = kb0;
                o[4] = kb1;
                o[5] = slot;
            }
            ++n;
        }
        return n;
    }
    const Work w = make_schedule(M, N, K, sm_count, passes);
    const int units = work_units(w);
    for (int u = 0; u < units && u < cap; ++u) {
        int tm, n0, nw, kb0, kb1, slot;
        unit_coords(w, u, tm, n0, nw, kb0, kb1, slot);
        int* o = out + 6 * size_t(u);
        o[0] = tm * BM;
        o[1] = n0;
        o[2] = nw;
        o[3] = kb0;
        o[4] = kb1;
        o[5] = slot;
    }
    return units;
}

size_t partial_bytes(int M, int N, int K, int sm_count, int passes) {
    if (passes == 1 && use_wide(M, N, K, sm_count))
        return wide_partial_bytes(make_wide_schedule(M, N, K, sm_count));
    const Work w = make_schedule(M, N, K, sm_count, passes);
    return size_t(w.splits) * w.split_tiles * BM * BN * sizeof(float);
}

constexpr size_t kCounterFloats = 512;  // the fused split's counters, 2 KiB
static_assert(kCounterFloats >= 1 + MAX_ROW_BLOCKS * MAX_SPLIT_CHUNKS && MAX_ROW_BLOCKS <= 32,
              "claim counter + one count per row block and chunk; row blocks fit a 32-bit mask");

size_t tc_workspace_bytes(int M, int N, int K, int passes, int sm_count, int chunk_rows,
                          bool raw_a) {
    const size_t planes = passes == 3 ? 2 : 1;
    const size_t a_planes = raw_a ? planes - 1 : planes;  // A itself is the hi plane
    size_t bytes = (a_planes * round_floats(size_t(M) * pad4(N)) +
                    planes * round_floats(size_t(K) * pad4(N)) + kCounterFloats) *
                   sizeof(float);
    if (chunk_rows <= 0 || chunk_rows >= M) return bytes + partial_bytes(M, N, K, sm_count, passes);
    // two sets: chunks alternate between two streams, so two chunk GEMMs may overlap
    return bytes + 2 * tc_partial_set_floats(M, N, K, passes, sm_count, chunk_rows) * sizeof(float);
}

size_t tc_partial_set_floats(int M, int N, int K, int passes, int sm_count, int chunk_rows) {
    size_t part = partial_bytes(chunk_rows, N, K, sm_count, passes);
    if (M % chunk_rows) {
        const size_t last = partial_bytes(M % chunk_rows, N, K, sm_count, passes);
        if (last > part) part = last;
    }
    return round_floats(part / sizeof(float));
}

TcLayout tc_layout(float* workspace, int M, int N, int K, int passes, const float* a_raw) {
    TcLayout L;
    L.lda = pad4(N);
    L.ldbt = pad4(N);
    L.a_raw = a_raw;
    const size_t a_plane = round_floats(size_t(M) * L.lda);
    const size_t b_plane = round_floats(size_t(K) * L.ldbt);
    // with a raw A there is no hi plane of A: a_hi is null and a_lo starts the workspace
    L.a_hi = a_raw ? nullptr : workspace;
    L.a_lo = passes == 3 ? (a_raw ? workspace : L.a_hi + a_plane) : L.a_hi;
    L.b_hi = passes == 3 ? L.a_lo + a_plane : L.a_hi + a_plane;
    L.b_lo = passes == 3 ? L.b_hi + b_plane : L.b_hi;
    L.counters = reinterpret_cast<int*>(L.b_lo + b_plane);
    L.partials = L.b_lo + b_plane + kCounterFloats;
    return L;
}

const float* tc_raw_hi(const float* A, int N, int passes) {
    return passes == 3 && N % 4 == 0 && aligned16(A) ? A : nullptr;
}

cudaError_t tc_prep(const float* A, int M, int a_row0, const float* B, int N, int K, int passes,
                    const TcLayout& L, int sm_count, cudaStream_t stream, const float* A_first,
                    int first_rows) {
    // (3xTF32 with a raw A: no hi plane, A itself is the GEMM's hi operand)
    float* a_hi = L.a_raw ? nullptr : L.a_hi + size_t(a_row0) * L.lda;
    float* a_lo = L.a_lo + size_t(a_row0) * L.lda;
    int a_blocks = 0, vec_a = 0;
    if (A) {
        vec_a = (N % 4 == 0 && aligned16(A)) ? 1 : 0;
        const size_t a_work = vec_a ? size_t(M) * N / 4 : size_t(M) * N;
        const size_t a_cap = size_t(sm_count > 0 ? sm_count : 1) * 8;
        a_blocks = int(a_work / 256 + 1 < a_cap ? a_work / 256 + 1 : a_cap);
    }
    const int b_tiles_k = (K + PREP_BT - 1) / PREP_BT;
    const int b_tiles = B ? b_tiles_k * ((N + PREP_BT - 1) / PREP_BT) : 0;
    PrepFirst first;
    if (A_first && B && first_rows > 0) {
        if (N % 4 != 0 || !aligned16(A_first) || L.lda != N) return cudaErrorInvalidValue;
        first.a = A_first;
        first.hi = passes == 3 ? (L.a_raw ? nullptr : L.a_hi) : L.a_hi;
        first.lo = passes == 3 ? L.a_lo : nullptr;
        first.rows = first_rows;
        first.n4 = N / 4;
        first.c4 = first.n4 < SPLIT_CHUNK4 ? first.n4 : SPLIT_CHUNK4;
        first.M = M;
        const int g = passes == 3 ? eager_rows_per_claim<2>() : eager_rows_per_claim<1>();
        first.claims = (first_rows + g - 1) / g;
        const size_t work = size_t(first_rows) * first.c4 / (256 * PREP_A_UNROLL) + 1;
        const size_t cap = size_t(sm_count > 0 ? sm_count : 1) * 4;
        first.blocks = int(work < cap ? work : cap);
    }
    if (a_blocks + first.blocks + b_tiles == 0) return cudaSuccess;
    // with B, the launch also sets the GEMM's counters (no GEMM on this workspace runs)
    int* zero = B ? L.counters : nullptr;
    const int grid = a_blocks + first.blocks + b_tiles;
    if (passes == 3)
        tf32_prep_kernel<2><<<grid, 256, 0, stream>>>(
            A, M, N, L.lda, a_hi, a_lo, vec_a, a_blocks, B, K, L.ldbt, L.b_hi, L.b_lo, b_tiles_k,
            zero, int(kCounterFloats), first);
    else
        tf32_prep_kernel<1><<<grid, 256, 0, stream>>>(
            A, M, N, L.lda, a_hi, nullptr, vec_a, a_blocks, B, K, L.ldbt, L.b_hi, nullptr,
            b_tiles_k, zero, int(kCounterFloats), first);
    count_launch();
    return cudaGetLastError();
}

cudaError_t tc_gemm_rows(const TcLayout& L, int row0, int rows, int N, int K, int passes,
                         float* C_rows, int sm_count, cudaStream_t stream,
                         const KernelTimer& timer, int* err, const float* A_fused) {
    // tensor maps over the planes: each CTA of a pair loads 32 x 128 boxes of A and of
    // B^T (its half of the tile's rows and of its columns)
    alignas(64) CUtensorMap ah, al, bh, bl;
    const float* a_hi = L.a_raw ? L.a_raw + size_t(row0) * N : L.a_hi + size_t(row0) * L.lda;
    const float* a_lo = L.a_lo + size_t(row0) * L.lda;
    if (L.a_raw && (passes != 3 || L.lda != N)) return cudaErrorInvalidValue;
    if (!encode_plane(&ah, a_hi, rows, N, L.lda, BK, HALF_M) ||
        !encode_plane(&bh, L.b_hi, K, N, L.ldbt, BK, HALF_N))
        return cudaErrorInvalidValue;
    if (passes == 3) {
        if (!encode_plane(&al, a_lo, rows, N, L.lda, BK, HALF_M) ||
            !encode_plane(&bl, L.b_lo, K, N, L.ldbt, BK, HALF_N))
            return cudaErrorInvalidValue;
    } else {
        al = ah;
        bl = bh;
    }
    const Work w = make_schedule(rows, N, K, sm_count, passes);
    FusedSplit fs{};
    if (A_fused) {
        if (N % 4 != 0 || !aligned16(A_fused) || L.lda != N) return cudaErrorInvalidValue;
        if (L.a_raw && A_fused != a_hi) return cudaErrorInvalidValue;  // A is the hi plane
        // the GEMM splits A's rows itself; B's pre-pass zeroed its counters
        fs.a = A_fused;
        fs.a_hi = L.a_raw ? nullptr : const_cast<float*>(a_hi);
        fs.a_lo = passes == 3 ? const_cast<float*>(a_lo) : nullptr;
        fs.counters = L.counters;
        fs.N = N;
        fs.chunks = (N / 4 + SPLIT_CHUNK4 - 1) / SPLIT_CHUNK4;
    }
    if (passes == 1 && use_wide(rows, N, K, sm_count))
        return launch_wide(ah, bh, C_rows, rows, N, K, L.partials, sm_count, stream, timer, err,
                           fs);
    // recut pieces load B^T in boxes of the widest piece's half-width
    alignas(64) CUtensorMap bph = bh, bpl = bl;
    if (w.pieces > 0) {
        if (!encode_plane(&bph, L.b_hi, K, N, L.ldbt, BK, w.piece_box)) return cudaErrorInvalidValue;
        if (passes == 3 && !encode_plane(&bpl, L.b_lo, K, N, L.ldbt, BK, w.piece_box))
            return cudaErrorInvalidValue;
        if (passes != 3) bpl = bph;
    }
    return passes == 3 ? launch_gemm<3>(ah, al, bh, bl, bph, bpl, C_rows, rows, N, K, w,
                                        L.partials, sm_count, stream, timer, err, fs)
                       : launch_gemm<1>(ah, al, bh, bl, bph, bpl, C_rows, rows, N, K, w,
                                        L.partials, sm_count, stream, timer, err, fs);
}

constexpr size_t kFuseMinElems = size_t(1) << 22;  // A of at least 16 MiB

cudaError_t launch_tc(const float* A, const float* B, float* C, int M, int N, int K, int passes,
                      float* workspace, int sm_count, cudaStream_t stream,
                      const KernelTimer& timer, int* err) {
    const TcLayout L = tc_layout(workspace, M, N, K, passes, tc_raw_hi(A, N, passes));
    // A large A with 16-byte rows whose first round of tiles reads less than half of its
    // rows: B is split first and A's split (3xTF32) or rounding (1xTF32) is fused into
    // the GEMM, where the rows of later rounds are prepared while earlier tiles are
    // multiplied. (Measured at 8192 x 6144 x 4096: +2.4 % for 3xTF32, +2.7 % for 1xTF32.
    // Where the first round reads most of A, as at 8192 x 8192 x 1024, fusing cost about
    // 1 %; with unaligned rows the few splitting warps fall behind the 1xTF32 GEMM.)
    const int pairs = sm_count / 2 > 0 ? sm_count / 2 : 1;
    const int first_rows =
        passes == 1 && use_wide(M, N, K, sm_count)
            ? first_round_rows_wide(make_wide_schedule(M, N, K, sm_count), M, pairs)
            : first_round_rows(make_schedule(M, N, K, sm_count, passes), M, pairs);
    const bool fuse = size_t(M) * N >= kFuseMinElems && N % 4 == 0 && aligned16(A) &&
                      2 * first_rows < M;
    // 1. round / split A (unless fused), transpose-round / split B into the padded planes
    cudaError_t e = tc_prep(fuse ? nullptr : A, M, 0, B, N, K, passes, L, sm_count, stream,
                            fuse ? A : nullptr, fuse ? first_rows : 0);
    if (e != cudaSuccess) return e;
    // 2. the GEMM over all rows
    return tc_gemm_rows(L, 0, M, N, K, passes, C, sm_count, stream, timer, err,
                        fuse ? A : nullptr);
}

cudaError_t tc_clock_record(cudaStream_t stream, unsigned long long (&out)[4]) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_clock_record, sizeof(out), 0,
                                              cudaMemcpyDeviceToHost, stream);
    return e == cudaSuccess ? cudaStreamSynchronize(stream) : e;
}

// ------------------------------------------------ FP16 three-product path (host) ----
// Workspace: A's hi and lo planes (M x pad8(N) halves each), B^T's (K x pad8(N)), the
// maxima of B's columns, the exponents of A's rows and B's columns, then the
// split-reduction partials.
// The schedule is the 3xTF32 one with 64 reduction elements per block.
namespace {
struct Tc16Layout {
    __half *a_hi, *a_lo, *b_hi, *b_lo;
    uint32_t* bmax;
    int *ea, *eb;
    float* partials;
    int ld;  // row pitch of every plane, halves
};

Tc16Layout tc16_layout(void* workspace, int M, int N, int K) {
    Tc16Layout L;
    L.ld = pad8(N);
    const size_t a_plane = round_halves(size_t(M) * L.ld), b_plane = round_halves(size_t(K) * L.ld);
    __half* h = static_cast<__half*>(workspace);
    L.a_hi = h;
    L.a_lo = h + a_plane;
    L.b_hi = h + 2 * a_plane;
    L.b_lo = h + 2 * a_plane + b_plane;
    L.bmax = reinterpret_cast<uint32_t*>(h + 2 * a_plane + 2 * b_plane);
    L.ea = reinterpret_cast<int*>(L.bmax + round_floats(size_t(K)));
    L.eb = L.ea + round_floats(size_t(M));
    L.partials = reinterpret_cast<float*>(L.eb + round_floats(size_t(K)));
    return L;
}

// the schedule of a product whose blocks hold 64 reduction elements
Work schedule16(int M, int N, int K, int sm_count) {
    return make_schedule(M, (N + 1) / 2, K, sm_count, 3);
}
}  // namespace

size_t tc16_workspace_bytes(int M, int N, int K, int sm_count) {
    const size_t planes = 2 * round_halves(size_t(M) * pad8(N)) + 2 * round_halves(size_t(K) * pad8(N));
    const size_t vecs = round_floats(size_t(M)) + 2 * round_floats(size_t(K));
    const Work w = schedule16(M, N, K, sm_count);
    return planes * sizeof(__half) + vecs * sizeof(uint32_t) +
           size_t(w.splits) * w.split_tiles * BM * BN * sizeof(float);
}

int tc16_schedule_units(int M, int N, int K, int sm_count, int* out, int cap) {
    return tc_schedule_units(M, (N + 1) / 2, K, 3, sm_count, out, cap);
}

cudaError_t launch_tc16(const float* A, const float* B, float* C, int M, int N, int K,
                        void* workspace, int sm_count, cudaStream_t stream,
                        const KernelTimer& timer, int* err) {
    const Tc16Layout L = tc16_layout(workspace, M, N, K);
    // 1. the maxima of B's column blocks
    cudaError_t e = cudaMemsetAsync(
        L.bmax, 0, size_t((K + F16_COL_BLOCK - 1) / F16_COL_BLOCK) * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    const int cap = (sm_count > 0 ? sm_count : 1) * 8;
    const int a_blocks = (M + 7) / 8 < cap ? (M + 7) / 8 : cap;
    const int b_cols = (K + 255) / 256;
    const int b_strips = (N + 31) / 32;
    // the maxima of B's 128-column blocks (the split finds each row's maximum of A itself)
    f16_colmax_kernel<<<b_cols * b_strips, 256, 0, stream>>>(B, N, K, b_cols, L.bmax);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 2. the scaled FP16 pieces
    const int b_tiles_k = (K + PREP_BT - 1) / PREP_BT;
    const int b_tiles = b_tiles_k * ((N + PREP_BT - 1) / PREP_BT);
    const int vec_a = (N % 4 == 0 && aligned16(A)) ? 1 : 0;
    f16_split_kernel<<<a_blocks + b_tiles, 256, 0, stream>>>(
        A, M, N, L.ld, L.a_hi, L.a_lo, a_blocks, vec_a, L.ea, B, K, L.ld, L.b_hi, L.b_lo,
        b_tiles_k, L.bmax, L.eb);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 3. the GEMM
    alignas(64) CUtensorMap ah, al, bh, bl;
    if (!encode_plane16(&ah, L.a_hi, M, N, L.ld, HALF_M) ||
        !encode_plane16(&al, L.a_lo, M, N, L.ld, HALF_M) ||
        !encode_plane16(&bh, L.b_hi, K, N, L.ld, HALF_N) ||
        !encode_plane16(&bl, L.b_lo, K, N, L.ld, HALF_N))
        return cudaErrorInvalidValue;
    const Work w = schedule16(M, N, K, sm_count);
    alignas(64) CUtensorMap bph = bh, bpl = bl;
    if (w.pieces > 0 && (!encode_plane16(&bph, L.b_hi, K, N, L.ld, w.piece_box) ||
                         !encode_plane16(&bpl, L.b_lo, K, N, L.ld, w.piece_box)))
        return cudaErrorInvalidValue;
    return launch_gemm<3, true>(ah, al, bh, bl, bph, bpl, C, M, N, K, w, L.partials, sm_count,
                                stream, timer, err, FusedSplit{}, L.ea, L.eb);
}

}  // namespace sgemm
