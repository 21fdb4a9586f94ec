// Kernels for layouts the TMA / tcgen05 kernel cannot take as they are:
// the repacking copy (below) and, first, the warp-level tensor-core path.
//
// Warp-level tensor-core path: mma.sync.aligned.m16n8k16 with register
// fragments, the lowering the TVM TIRx "gemm" page describes (sections
// "Demonstration program", "Algorithm" and "Generated CUDA"), used for the
// cases the TMA / tcgen05 kernel cannot take or does not pay off for:
//
//  * operands or outputs whose addresses or row strides are not 16-byte
//    multiples (TMA cannot describe them; this path loads element by
//    element, so any element-aligned layout works);
//  * tiny problems, where the tcgen05 kernel's set-up (tensor memory,
//    barriers, TMA descriptors) costs more than the arithmetic.
//
// Fragment layout of one m16n8k16 atom, lane = 4 g + t (g = lane / 4,
// t = lane % 4), exactly as the demonstration program stages it:
//   A (16 x 16): slot s = 4 kHi + 2 rM + kp holds A[g + 8 rM][2 t + kp + 8 kHi]
//                (the slot order of the TIRx gemm guide, section 三; the
//                 operand registers a0..a3 pack slot pairs (kp = 0, 1))
//   B (16 x 8):  slot s = 2 kHi + kp holds B[2 t + kp + 8 kHi][g]
//   D (16 x 8):  slot s = 2 rM + rN holds D[g + 8 rM][2 t + rN]
// D is initialised to 0 and accumulated over K in place (TIRx "Algorithm",
// step 3); alpha and beta are applied in the epilogue like the tcgen05 path.
// K is covered by k16 atoms; a remainder of at most 8 takes one m16n8k8
// atom, as the lowering does for K = 8 (mod 16).  Staged columns past K are
// zero, so the last k16 atom of a ragged K adds nothing for them.
//
// Two kernels share this lowering:
//  * gemm_mma_sync_kernel: CTA tile 128 x 128, 8 warps in a 2 x 4 grid of
//    64 x 32 warp tiles (4 x 4 atoms each); K slabs of 32 double-buffered in
//    shared memory with padded rows, the next slab's loads in flight during
//    the current MMAs.  For layouts TMA cannot take, at any size.
//  * gemm_mma_atom_kernel: one warp per 16 x 8 block of D (one atom wide),
//    its fragments read straight from global memory into the slots above --
//    the demonstration program's own shape, with no shared staging and no
//    CTA barrier.  For tiny problems, whose time is the launch and a chain
//    of memory latencies: a 16 x 8 x 16 product takes 1.6 us per launch
//    (graph-replayed) against 4.1 us for the tiled kernel's 256-thread CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_internal.h"
#include "ptx.cuh"

namespace gb300 {

namespace {

constexpr int kSBM = 128, kSBN = 128, kSBK = 32;   // CTA tile and K slab
constexpr int kSThreads = 256;                     // 8 warps in a 2 (M) x 4 (N) grid
constexpr int kWarpsN = 4;
constexpr int kWarpM = 64, kWarpN = 32;            // warp tile
constexpr int kAtomsM = kWarpM / 16, kAtomsN = kWarpN / 8;
constexpr int kPad = 8;   // halves of padding per shared row (conflict-free fragment loads)
static_assert(kSBM / kWarpM * (kSBN / kWarpN) == kSThreads / 32, "one warp tile per warp");

template <int kIn>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    if constexpr (kIn == 0)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// m16n8k8: the atom for a K remainder of 8 (the lowering's k8 shape).  Its
// A fragment is the kHi = 0 half of the k16 one (slots rM = 0, 1), its B
// fragment the kHi = 0 register.
template <int kIn>
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    if constexpr (kIn == 0)
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(b0));
}

__device__ __forceinline__ uint32_t pack_halves(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

template <int kOut>
__device__ __forceinline__ float load_out(const void* p, int64_t i) {
    if constexpr (kOut == kOutF32) return static_cast<const float*>(p)[i];
    if constexpr (kOut == kOutF16) return __half2float(static_cast<const __half*>(p)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

template <int kOut>
__device__ __forceinline__ void store_out(void* p, int64_t i, float v) {
    if constexpr (kOut == kOutF32)
        static_cast<float*>(p)[i] = v;
    else if constexpr (kOut == kOutF16)
        static_cast<__half*>(p)[i] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// Operand staging: the slab [rows, kSBK] of one operand, read element by
// element (any element-aligned layout) with consecutive threads on the
// operand's contiguous dimension, into registers; out-of-range -> 0.
//   trans = 0: element (r, k) at X[(r0 + r) * ld + k0 + k]   (K contiguous)
//   trans = 1: element (r, k) at X[(k0 + k) * ld + r0 + r]   (rows contiguous)
template <int kRows>
__device__ __forceinline__ void load_slab(uint16_t (&v)[kRows * kSBK / kSThreads], const uint16_t* X, int trans,
                                          int64_t ld, int64_t r0, int64_t rows, int64_t k0, int64_t K) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < kRows * kSBK / kSThreads; ++i) {
        const int e = tid + i * kSThreads;
        const int r = trans ? e % kRows : e / kSBK;
        const int c = trans ? e / kRows : e % kSBK;
        const int64_t rr = r0 + r, kk = k0 + c;
        v[i] = (rr < rows && kk < K) ? (trans ? X[kk * ld + rr] : X[rr * ld + kk]) : (uint16_t)0;
    }
}

// ... and from registers into the K-contiguous shared slab S[r][k].
template <int kRows>
__device__ __forceinline__ void store_slab(uint16_t (*S)[kSBK + kPad], const uint16_t (&v)[kRows * kSBK / kSThreads],
                                           int trans) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < kRows * kSBK / kSThreads; ++i) {
        const int e = tid + i * kSThreads;
        const int r = trans ? e % kRows : e / kSBK;
        const int c = trans ? e / kRows : e % kSBK;
        S[r][c] = v[i];
    }
}

// One kSBM x kSBN tile of D at (m0, n0).  The K loop is software-pipelined:
// the next slab's global loads are in flight (in registers) while the
// current slab, double-buffered in shared memory, feeds the MMAs.
template <int kIn, int kOut, bool kHasC>
__device__ __forceinline__ void sync_tile(const SyncParams& p, int64_t m0, int64_t n0,
                                          uint16_t (*As)[kSBM][kSBK + kPad], uint16_t (*Bs)[kSBN][kSBK + kPad]) {
    const int tid = threadIdx.x;
    const int lane = tid % 32;
    const int warp = tid / 32;
    const int g = lane / 4, tq = lane % 4;
    const int wm = (warp / kWarpsN) * kWarpM, wn = (warp % kWarpsN) * kWarpN;   // warp tile origin
    const uint16_t* A = static_cast<const uint16_t*>(p.A);
    const uint16_t* B = static_cast<const uint16_t*>(p.B);
    // B as [N rows][K]: transB = 1 is K-contiguous, transB = 0 (stored [K, N]) rows-contiguous
    const int b_trans = p.transB ? 0 : 1;

    float acc[kAtomsM][kAtomsN][4];
#pragma unroll
    for (int i = 0; i < kAtomsM; ++i)
#pragma unroll
        for (int j = 0; j < kAtomsN; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) acc[i][j][s] = 0.0f;

    uint16_t ra[kSBM * kSBK / kSThreads], rb[kSBN * kSBK / kSThreads];
    load_slab<kSBM>(ra, A, p.transA, p.lda, m0, p.M, 0, p.K);
    load_slab<kSBN>(rb, B, b_trans, p.ldb, n0, p.N, 0, p.K);
    store_slab<kSBM>(As[0], ra, p.transA);
    store_slab<kSBN>(Bs[0], rb, b_trans);
    __syncthreads();
    int cur = 0;
    for (int64_t k0 = 0; k0 < p.K; k0 += kSBK) {
        const bool more = k0 + kSBK < p.K;   // the same for the whole CTA
        if (more) {
            load_slab<kSBM>(ra, A, p.transA, p.lda, m0, p.M, k0 + kSBK, p.K);
            load_slab<kSBN>(rb, B, b_trans, p.ldb, n0, p.N, k0 + kSBK, p.K);
        }
#pragma unroll
        for (int ks = 0; ks < kSBK; ks += 16) {
            const int64_t k_left = p.K - (k0 + ks);   // same for the whole CTA
            if (k_left <= 0) break;
            uint32_t af[kAtomsM][4], bf[kAtomsN][2];
#pragma unroll
            for (int i = 0; i < kAtomsM; ++i) {
                const int r = wm + 16 * i + g;
#pragma unroll
                for (int w = 0; w < 4; ++w) {   // w = 2 kHi + rM: slots 2w, 2w + 1 (kp = 0, 1)
                    const int rM = w % 2, kHi = w / 2;
                    const int c = ks + 2 * tq + 8 * kHi;
                    af[i][w] = pack_halves(As[cur][r + 8 * rM][c], As[cur][r + 8 * rM][c + 1]);
                }
            }
#pragma unroll
            for (int j = 0; j < kAtomsN; ++j) {
                const int r = wn + 8 * j + g;
#pragma unroll
                for (int kHi = 0; kHi < 2; ++kHi) {   // slots 2 kHi, 2 kHi + 1
                    const int c = ks + 2 * tq + 8 * kHi;
                    bf[j][kHi] = pack_halves(Bs[cur][r][c], Bs[cur][r][c + 1]);
                }
            }
            if (k_left > 8) {
#pragma unroll
                for (int i = 0; i < kAtomsM; ++i)
#pragma unroll
                    for (int j = 0; j < kAtomsN; ++j) mma_16816<kIn>(acc[i][j], af[i], bf[j]);
            } else {   // at most 8 columns of K left: one k8 atom
#pragma unroll
                for (int i = 0; i < kAtomsM; ++i)
#pragma unroll
                    for (int j = 0; j < kAtomsN; ++j) mma_1688<kIn>(acc[i][j], af[i][0], af[i][1], bf[j][0]);
            }
        }
        if (more) {   // the other buffer was last read before the previous barrier
            store_slab<kSBM>(As[cur ^ 1], ra, p.transA);
            store_slab<kSBN>(Bs[cur ^ 1], rb, b_trans);
        }
        __syncthreads();
        cur ^= 1;
    }

    // epilogue: D = alpha * acc (+ beta * C), element by element with bounds
#pragma unroll
    for (int i = 0; i < kAtomsM; ++i)
#pragma unroll
        for (int j = 0; j < kAtomsN; ++j)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int rM = s / 2, rN = s % 2;
                const int64_t m = m0 + wm + 16 * i + g + 8 * rM;
                const int64_t n = n0 + wn + 8 * j + 2 * tq + rN;
                if (m < p.M && n < p.N) {
                    float d;
                    if constexpr (kHasC)
                        d = fmaf(p.alpha, acc[i][j][s], p.beta * load_out<kOut>(p.C, m * p.ldc + n));
                    else
                        d = p.alpha * acc[i][j][s];
                    store_out<kOut>(p.D, m * p.ldd + n, d);
                }
            }
}

template <int kIn, int kOut, bool kHasC>
__global__ void __launch_bounds__(kSThreads) gemm_mma_sync_kernel(SyncParams p) {
    // As[buf][m][k] and Bs[buf][n][k]: both K-contiguous, so A and B
    // fragments are read the same way (pairs of consecutive k).
    __shared__ uint16_t As[2][kSBM][kSBK + kPad];
    __shared__ uint16_t Bs[2][kSBN][kSBK + kPad];
    ptx::grid_dependency_wait();   // the previous kernel's writes are visible (programmatic launch)
    ptx::launch_dependents();
    const int64_t num_m_tiles = (p.M + kSBM - 1) / kSBM;
    // grid.y is capped at 65535: CTAs step through the M tiles by gridDim.y
    for (int64_t mt = blockIdx.y; mt < num_m_tiles; mt += gridDim.y) {
        sync_tile<kIn, kOut, kHasC>(p, mt * kSBM, (int64_t)blockIdx.x * kSBN, As, Bs);
        __syncthreads();   // the next tile's first stores must not overtake this tile's reads
    }
}

constexpr int kAtomWarps = 4;   // warps per CTA of the atom kernel
// K steps (of 16) whose fragments the atom kernel loads together: 1 for
// K <= 32, where the extra predicated loads of a longer group cost more than
// they hide (16x8x16: 1.6 vs 2.1 us per launch), else 4 (16x16x4096: 150 vs
// 183 us; 128^3: 6.2 vs 7.3 us; graph-replayed on GB300)
constexpr int kAtomStepsDeep = 4;
constexpr int64_t kAtomShallowK = 32;

// D = alpha * op(A) @ op(B) (+ beta * C) one 16 x 8 block per warp.  Lane
// 4 g + t loads its A slots (rows g, g + 8; K columns 2 t, 2 t + 1 and
// 8 more) and B slots (column g; the same K rows) from global memory,
// out-of-range elements as 0, so a ragged M, N or K needs no other care;
// a K remainder of at most 8 takes the m16n8k8 atom, as in the tiled kernel.
template <int kIn, int kOut, bool kHasC, int kSteps>
__global__ void __launch_bounds__(kAtomWarps * 32) gemm_mma_atom_kernel(SyncParams p) {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    const int lane = threadIdx.x % 32;
    const int g = lane / 4, tq = lane % 4;
    const uint16_t* A = static_cast<const uint16_t*>(p.A);
    const uint16_t* B = static_cast<const uint16_t*>(p.B);
    const int64_t n_blocks = (p.N + 7) / 8;
    const int64_t blocks = (p.M + 15) / 16 * n_blocks;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    // element steps of op(A) along its rows (M) and along K, and of op(B)
    // along K and its columns (N)
    const int64_t a_sm = p.transA ? 1 : p.lda, a_sk = p.transA ? p.lda : 1;
    const int64_t b_sk = p.transB ? 1 : p.ldb, b_sn = p.transB ? p.ldb : 1;
    for (int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; blk < blocks; blk += warps) {
        const int64_t m0 = blk / n_blocks * 16, n0 = blk % n_blocks * 8;
        // this lane's rows of op(A) (g, g + 8) and column of op(B) (g)
        const bool in_r0 = m0 + g < p.M, in_r1 = m0 + g + 8 < p.M, in_n = n0 + g < p.N;
        const uint16_t* a_r0 = A + (in_r0 ? (m0 + g) * a_sm : 0);
        const uint16_t* a_r1 = A + (in_r1 ? (m0 + g + 8) * a_sm : 0);
        const uint16_t* b_n = B + (in_n ? (n0 + g) * b_sn : 0);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        // kSteps K steps at a time: all their fragment loads are issued
        // (predicated, with no branch between them) before the first of
        // their MMAs, so the steps share one memory latency instead of paying
        // one each.  Steps past K load nothing.
        for (int64_t kc = 0; kc < p.K; kc += 16 * kSteps) {
            const int64_t left = p.K - kc;   // the same for the whole warp
            uint32_t af[kSteps][4], bf[kSteps][2];
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
#pragma unroll
                for (int kHi = 0; kHi < 2; ++kHi) {
                    const int64_t k = kc + 16 * st + 2 * tq + 8 * kHi;   // K columns k, k + 1
                    const bool k0_in = k < p.K, k1_in = k + 1 < p.K;
                    // A slots: w = 2 kHi + rM, as in the tiled kernel
                    af[st][2 * kHi] = pack_halves(in_r0 && k0_in ? a_r0[k * a_sk] : (uint16_t)0,
                                                  in_r0 && k1_in ? a_r0[(k + 1) * a_sk] : (uint16_t)0);
                    af[st][2 * kHi + 1] = pack_halves(in_r1 && k0_in ? a_r1[k * a_sk] : (uint16_t)0,
                                                      in_r1 && k1_in ? a_r1[(k + 1) * a_sk] : (uint16_t)0);
                    bf[st][kHi] = pack_halves(in_n && k0_in ? b_n[k * b_sk] : (uint16_t)0,
                                              in_n && k1_in ? b_n[(k + 1) * b_sk] : (uint16_t)0);
                }
            }
#pragma unroll
            for (int st = 0; st < kSteps; ++st) {
                const int64_t k_left = left - 16 * st;
                if (k_left <= 0) break;
                if (k_left > 8)
                    mma_16816<kIn>(acc, af[st], bf[st]);
                else
                    mma_1688<kIn>(acc, af[st][0], af[st][1], bf[st][0]);
            }
        }
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int64_t m = m0 + g + 8 * (s / 2);
            const int64_t n = n0 + 2 * tq + s % 2;
            if (m < p.M && n < p.N) {
                float d;
                if constexpr (kHasC)
                    d = fmaf(p.alpha, acc[s], p.beta * load_out<kOut>(p.C, m * p.ldc + n));
                else
                    d = p.alpha * acc[s];
                store_out<kOut>(p.D, m * p.ldd + n, d);
            }
        }
    }
}

template <int kIn, int kOut, bool kHasC>
cudaError_t launch_sync_one(const SyncParams& p, cudaStream_t stream) {
    if (p.atom) {
        const int64_t blocks = (p.M + 15) / 16 * ((p.N + 7) / 8);
        const int64_t warps = blocks < kAtomWarps ? blocks : kAtomWarps;
        const int64_t ctas = (blocks + warps - 1) / warps;
        const dim3 grid((unsigned)(ctas < 65535 ? ctas : 65535)), block((unsigned)(32 * warps));
        if (p.K <= kAtomShallowK) return launch_with_pdl(gemm_mma_atom_kernel<kIn, kOut, kHasC, 1>, grid, block, stream, p);
        return launch_with_pdl(gemm_mma_atom_kernel<kIn, kOut, kHasC, kAtomStepsDeep>, grid, block, stream, p);
    }
    const int64_t m_tiles = (p.M + kSBM - 1) / kSBM;
    const dim3 grid((unsigned)((p.N + kSBN - 1) / kSBN), (unsigned)(m_tiles < 65535 ? m_tiles : 65535));
    return launch_with_pdl(gemm_mma_sync_kernel<kIn, kOut, kHasC>, grid, dim3(kSThreads), stream, p);
}

template <int kIn, bool kHasC>
cudaError_t launch_sync_out(const SyncParams& p, cudaStream_t stream) {
    if (p.out == kOutF32) return launch_sync_one<kIn, kOutF32, kHasC>(p, stream);
    if (p.out == kOutF16) return launch_sync_one<kIn, kOutF16, kHasC>(p, stream);
    return launch_sync_one<kIn, kOutBF16, kHasC>(p, stream);
}

// Row-major 2-D copy between element-aligned layouts with any row strides:
// the repacking step that gives the tcgen05 kernel's TMA copies 16-byte-
// aligned operands and outputs.  Consecutive threads take consecutive
// elements of a row.
template <typename T>
__global__ void copy2d_kernel(T* dst, int64_t ldd, const T* src, int64_t lds, int64_t rows, int64_t cols) {
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y)
        for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < cols;
             c += (int64_t)gridDim.x * blockDim.x)
            dst[r * ldd + c] = src[r * lds + c];
}

// dst[c * ldd + r] = src[r * lds + c] for r < rows, c < cols: the
// repacking step that turns an 8-bit operand stored MN-major into the
// K-major copy the tcgen05 kernel stages.  32 x 32 tiles through shared
// memory, so that both the reads and the writes walk rows.
constexpr int kTT = 32;
template <typename T>
__global__ void transpose2d_kernel(T* dst, int64_t ldd, const T* src, int64_t lds, int64_t rows, int64_t cols) {
    __shared__ T tile[kTT][kTT + 1];
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    const int64_t tiles_r = (rows + kTT - 1) / kTT, tiles_c = (cols + kTT - 1) / kTT;
    for (int64_t br = blockIdx.y; br < tiles_r; br += gridDim.y)
        for (int64_t bc = blockIdx.x; bc < tiles_c; bc += gridDim.x) {
            const int64_t r0 = br * kTT, c0 = bc * kTT;
            for (int i = threadIdx.y; i < kTT; i += blockDim.y) {
                const int64_t r = r0 + i, c = c0 + threadIdx.x;
                if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * lds + c];
            }
            __syncthreads();
            for (int i = threadIdx.y; i < kTT; i += blockDim.y) {
                const int64_t c = c0 + i, r = r0 + threadIdx.x;   // dst row c, column r
                if (r < rows && c < cols) dst[c * ldd + r] = tile[threadIdx.x][i];
            }
            __syncthreads();
        }
}

}  // namespace

cudaError_t launch_mma_sync(const SyncParams& p, cudaStream_t stream) {
    if (p.in_bf16) return p.has_c ? launch_sync_out<1, true>(p, stream) : launch_sync_out<1, false>(p, stream);
    return p.has_c ? launch_sync_out<0, true>(p, stream) : launch_sync_out<0, false>(p, stream);
}

cudaError_t launch_copy2d(void* dst, int64_t ldd, const void* src, int64_t lds, int64_t rows, int64_t cols,
                          int elem_bytes, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    constexpr int kThreads = 256;
    int64_t gx = (cols + kThreads - 1) / kThreads;
    if (gx > 64) gx = 64;
    const int64_t gy = rows < 65535 ? rows : 65535;
    const dim3 grid((unsigned)gx, (unsigned)gy);
    if (elem_bytes == 4)
        return launch_with_pdl(copy2d_kernel<uint32_t>, grid, dim3(kThreads), stream, static_cast<uint32_t*>(dst),
                               ldd, static_cast<const uint32_t*>(src), lds, rows, cols);
    if (elem_bytes == 2)
        return launch_with_pdl(copy2d_kernel<uint16_t>, grid, dim3(kThreads), stream, static_cast<uint16_t*>(dst),
                               ldd, static_cast<const uint16_t*>(src), lds, rows, cols);
    return launch_with_pdl(copy2d_kernel<uint8_t>, grid, dim3(kThreads), stream, static_cast<uint8_t*>(dst), ldd,
                           static_cast<const uint8_t*>(src), lds, rows, cols);
}

cudaError_t launch_transpose2d(void* dst, int64_t ldd, const void* src, int64_t lds, int64_t rows, int64_t cols,
                               int elem_bytes, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int64_t tr = (rows + kTT - 1) / kTT, tc = (cols + kTT - 1) / kTT;
    const dim3 grid((unsigned)(tc < 65535 ? tc : 65535), (unsigned)(tr < 65535 ? tr : 65535));
    const dim3 block(kTT, kTT / 4);
    if (elem_bytes == 2)
        return launch_with_pdl(transpose2d_kernel<uint16_t>, grid, block, stream, static_cast<uint16_t*>(dst), ldd,
                               static_cast<const uint16_t*>(src), lds, rows, cols);
    return launch_with_pdl(transpose2d_kernel<uint8_t>, grid, block, stream, static_cast<uint8_t*>(dst), ldd,
                           static_cast<const uint8_t*>(src), lds, rows, cols);
}

}  // namespace gb300
