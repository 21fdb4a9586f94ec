// The sm_103a tcgen05 kernel for D = alpha * op(A) @ op(B) + beta * C, as a
// template included by the translation units that instantiate it
// (gemm_sm103.cu: fp16 / bf16 operands; gemm_sm103_f8.cu: E4M3 / E5M2).
//
// The contraction is the one of the TVM TIRx "gemm" page (opening paragraph
// and "What it accepts": f16/bf16 operands, f32 accumulator, D initialised
// to 0 for beta = 0 or from C for beta = 1) with the general epilogue
// alpha * acc + beta * c_old of the Phobos "@tensorcore" page
// (gemm_fp16tc_fp32acc.ph).  The pages lower it to warp-level mma.sync
// fragments in registers; here it is re-designed for Blackwell:
//
//  * operand staging: TMA 2-D tile loads into 128-byte-swizzled shared
//    memory, an S-stage full/empty mbarrier ring (replaces the pages'
//    swizzled cp.async staging, Phobos "@tensorcore" page, section
//    "Interactions", @pipeline);
//  * main loop: tcgen05.mma kind::f16 (fp16 / bf16) or kind::f8f6f4 (the
//    8-bit precisions the TIRx gemm guide lists for the tcgen05 path,
//    section 七) issued by one thread, accumulator in
//    tensor memory (TMEM), the first K step with the accumulate flag off
//    (the TIRx "Algorithm" step 3 "initialise D, then accumulate over K in
//    place" becomes "overwrite, then accumulate");
//  * warp specialisation: warp 0 = TMA producer, warp 1 = TMEM allocator
//    and MMA issuer, warps 2..5 = epilogue (one TMEM lane quadrant each);
//  * two accumulators in TMEM (2 x 256 columns) so the epilogue of tile i
//    overlaps the main loop of tile i+1;
//  * persistent grid with grouped (L2-friendly) tile order;
//  * optional CTA pair (cta_group::2): a 256 x 256 tile per cluster of two
//    SMs, each SM loading its half of A and its half of B;
//  * epilogue: tcgen05.ld TMEM -> registers, alpha/beta (C fetched by TMA
//    only when beta != 0), conversion, swizzled shared staging, TMA store;
//  * masked edges: TMA zero-fills out-of-range operand elements and clips
//    out-of-range stores, so ragged M, N, K need no separate path;
//  * every wait is bounded by the global timer; a wait that gives up records
//    itself in a device status block and the kernel unwinds cleanly.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_internal.h"
#include "gemm_params.h"
#include "ptx.cuh"

namespace gb300 {

constexpr int kBM = 128;             // accumulator rows per CTA (= TMEM lanes)
constexpr int kBNMax = 256;          // accumulator columns of the throughput tiles
constexpr int kNarrowN = 64;         // accumulator columns of the narrow (small-problem) tiles
constexpr int kFitN = 224;           // wave-fitted CTA-pair tiles: f32 D, K-major B only
constexpr int kBK = 64;              // K per sub-block: one 128-byte swizzle row of 16-bit elements
constexpr int kUK = 16;              // K per tcgen05.mma kind::f16
constexpr int kBK8 = 128;            // the same for 8-bit elements
constexpr int kUK8 = 32;             // K per tcgen05.mma kind::f8f6f4 (32 bytes, like kUK 16-bit elements)
constexpr int kEpiBufBytes = 4096;   // one epilogue staging box: 32 rows x 128 bytes
constexpr int kTmemCols = 512;       // two accumulators of up to 128 x 256 fp32
constexpr int kAtomBytes = 1024;     // 8 rows x 128 bytes: one 128B-swizzle atom
constexpr int kMnChunkBytes = 64 * kBK * 2;   // one 64-wide MN-major box (64 x 64 x 2 B)
constexpr int kSmemBudget = 232448;  // dynamic shared memory per CTA on sm_103
static_assert(kBK / kUK == 4, "the MMA loop issues four K slices per stage");
// MX block-scaled 8-bit operands: one UE8M0 scale per 32 K elements of each
// row of A and column of B.  A 128-K sub-block spans four scale blocks, so
// each row's scales of a sub-block are one 32-bit word.  Tiles are 224
// columns wide for f32 D and 192 for 16-bit D (on one SM or a CTA pair):
// two accumulators take 448 or 384 TMEM columns, scale slots the rest.
constexpr int kMxBlock = 32;         // K elements per scale
constexpr int kMxTileN = 192;        // accumulator columns of the block-scaled tiles (16-bit D)
constexpr int kMxTileNF32 = 224;     // the same for f32 D, whose 32-column epilogue chunks allow it
constexpr int kSfChunkBytes = 512;   // scales of 128 rows x 4 blocks, in tcgen05.cp order
constexpr int kSfSlotCols = 16;      // TMEM columns per sub-block's scales: SFA 4, SFB 4 per 128 columns of N
static_assert(kBK8 == 4 * kMxBlock, "one scale word per row and stage");

// kEpiW epilogue warps: 4 (one per TMEM lane quadrant, each storing all
// columns of its 32 rows) for K-heavy shapes, or 8 (two per quadrant, half
// the columns each) for shapes whose time goes into storing D; the operand
// ring gets whatever shared memory the staging boxes leave.
// kTileN: 256 (the throughput tiles: 256 x 256 per CTA pair, 128 x 256 per
// single CTA), 224 (256 x 224 CTA-pair tiles, f32 D and K-major B, for
// shapes whose 256-wide tiles leave the last wave mostly empty: 4096^2
// gives 256 tiles = 3.4 waves of 76 pairs at 256 wide, 304 = 4.0 at 224)
// or 64 (128 x 64 single-CTA tiles for problems too small to fill the GPU
// with wide tiles: four times as many CTAs, each with a quarter of the
// epilogue).
// kMX: the block-scaled variant (8-bit K-major operands): each sub-block of a
// stage also carries the scales of the CTA's 128 rows of A and of all kTileN
// columns of B (both CTAs of a pair need every column's scales), and two
// accumulators plus the scale slots share the 512 TMEM columns.
template <bool kPair, int kEpiW, int kTileN_ = kBNMax, bool kMX_ = false>
struct Cfg {
    static constexpr int kTileN = kTileN_;                 // D columns per tile
    static constexpr bool kMX = kMX_;
    static constexpr int kCtaGroup = kPair ? 2 : 1;
    static constexpr int kTileM = kPair ? 2 * kBM : kBM;   // D rows per tile
    static constexpr int kLoadN = kPair ? kTileN / 2 : kTileN;   // B rows (N) each CTA stages
    static constexpr int kEpiWarps = kEpiW;
    // producer, MMA, epilogue warps (+ kMX: the warp that copies the scales)
    static constexpr int kNumThreads = 64 + 32 * kEpiW + (kMX ? 32 : 0);
    static constexpr int kEpiCols = kTileN / (kEpiW / 4);  // accumulator columns per epilogue warp
    // MN-major B is staged in 64-wide boxes; the 224-wide and block-scaled
    // tiles (112 or 96 B rows per CTA) are launched for K-major B only.
    static_assert(kMX || kTileN == kFitN || kLoadN % 64 == 0, "MN-major operand boxes are 64 wide");
    static_assert(kTileN <= kBNMax && kTileN % ((kMX || kTileN == kFitN) ? 32 : 64) == 0, "tile width");
    // A pipeline stage holds kSub 64-wide K sub-blocks.  The MMA issuer pays a
    // fixed cost per stage (barrier wait, release commit) while the tensor
    // core queues only a few MMAs, so the pair kernel puts 8 MMAs (2 sub-
    // blocks) behind each wait: 64 KiB stages instead of 32 KiB ones.  The
    // 8-epilogue-warp kernel (tiles of a few stages, bound by the D stores)
    // keeps 32 KiB stages: beside its staging boxes that makes four stages
    // instead of two, so the loads of the next tile start sooner.  The
    // narrow 128 x 64 tiles take two sub-blocks per stage too (four 48 KiB
    // stages), so that a whole stage of each operand arrives in one TMA copy
    // (512^3: 6.4 -> 5.7 us per call).
    static constexpr int kSub = (kEpiW == 4 && (kPair || kTileN == kNarrowN)) ? 2 : 1;
    static constexpr int kASubBytes = kBM * kBK * 2;
    static constexpr int kBSubBytes = kLoadN * kBK * 2;
    static constexpr int kABytes = kSub * kASubBytes;
    static constexpr int kBBytes = kSub * kBSubBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    // staging boxes per epilogue warp: the store-bound configuration keeps
    // more D bytes in flight per SM
    static constexpr int kEpiBufs = kEpiW == 8 ? 3 : 2;
    static constexpr int kEpiBytes = kEpiW * kEpiBufs * kEpiBufBytes;
    // scales of one stage (kMX): per sub-block, SFA of the CTA's 128 rows,
    // then SFB in 128-column groups
    static constexpr int kSfbChunks = (kTileN + 127) / 128;
    static constexpr int kSfSubBytes = (1 + kSfbChunks) * kSfChunkBytes;
    static constexpr int kSfBytes = kMX ? kSub * kSfSubBytes : 0;
    static constexpr int kSfStageCols = kSub * kSfSlotCols;   // TMEM columns of one stage's scales
    static constexpr int kStages = (kSmemBudget - kEpiBytes - 2048 - (kMX ? 1024 : 0)) / (kStageBytes + kSfBytes);
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffSf = kOffB + kStages * kBBytes;
    static constexpr int kOffEpi = kOffSf + (kStages * kSfBytes + 1023) / 1024 * 1024;
    static constexpr int kOffBar = kOffEpi + kEpiBytes;
    // full[S], empty[S], tmem_full[2], tmem_empty[2], c_ready[epilogue warps][kEpiBufs],
    // kMX: scales_ready[S]
    static constexpr int kNumBars = 2 * kStages + 4 + kEpiBufs * kEpiW + (kMX ? kStages : 0);
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffSkFlag = kOffAbort + 4;    // "this CTA finishes the stream-K tile"
    static constexpr int kSmemBytes = kOffSkFlag + 4 + 1024;   // + base alignment slack
    static_assert(kStages >= 2, "at least two operand stages");
    static_assert(kSmemBytes <= kSmemBudget, "shared memory budget");
    // One TMEM scale slot per operand stage (see the MMA issuer).
    // TMEM scale slots (one stage's scales each) beside the two accumulators:
    // one per stage when they fit, else a ring the scale warp reuses once the
    // MMAs that read a slot have committed.
    static constexpr int kSfSlotsFit = kMX ? (kTmemCols - 2 * kTileN) / kSfStageCols : 1;
    static constexpr int kSfSlots = kSfSlotsFit < kStages ? kSfSlotsFit : kStages;
    static_assert(!kMX || (kSfSlots >= 2 && 2 * kTileN + kSfSlots * kSfStageCols <= kTmemCols &&
                           4 + 4 * kSfbChunks <= kSfSlotCols),
                  "block-scaled tiles: accumulators and scale slots within the TMEM allocation");
};

// tcgen05 shared-memory matrix descriptor for a 128-byte-swizzled operand:
// start address, leading / stride byte offsets (all >> 4), the fixed
// descriptor version 0b001 at bits 46-48, base offset 0, swizzle mode 2
// (128 B) at bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

// Descriptor of the kk-th K=16 slice of a staged operand tile.
//  K-major (K contiguous): rows of 128 B, 8-row atoms 1024 B apart (SBO);
//    a K step of 16 elements is +32 B inside the swizzle row.
//  MN-major (M or N contiguous): boxes of 64 MN x 64 K, each K row 128 B;
//    8-K-row atoms 1024 B apart (SBO), 64-wide MN boxes 8 KiB apart (LBO);
//    a K step of 16 rows is +2 KiB.
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile, int mn_major, int kk) {
    return mn_major ? sw128_desc(tile + kk * (kUK * 128), kMnChunkBytes, kAtomBytes)
                    : sw128_desc(tile + kk * (kUK * 2), 16, kAtomBytes);
}

// Descriptor of one 512-byte scale chunk for tcgen05.cp (no swizzle): 32
// rows of 16 bytes, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
           (1ull << 46);
}

static __device__ __noinline__ void report_timeout(const GemmParams& p, int site, int detail) {
    if (atomicCAS(&p.status->code, 0, kDeviceErrTimeout) == 0) {
        p.status->block = blockIdx.x;
        p.status->site = site;
        p.status->detail = detail;
        __threadfence();
    }
}

// Wait for the phase of `bar` with parity `parity`; gives up (returns false)
// when another thread of the CTA has aborted or the time bound has passed.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                             const GemmParams& p, int site, int detail) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0) {
            if (*abort) return false;
            if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
                *abort = 1;
                report_timeout(p, site, detail);
                return false;
            }
        }
    }
}

// Barrier among the epilogue warps only (named barrier 1; barrier 0 is
// __syncthreads).
template <int kEpiW>
__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiW * 32) : "memory");
}

// Counts one contributor into a stream-K tile and tells whether it is the
// last of `nc`.  The counter word holds (launch epoch << 8) | count, so a
// word left behind by an earlier or interrupted launch restarts at 1 instead
// of being trusted.  The retry loop is bounded (each failure means another
// contributor succeeded); if it runs out the CTA aborts.
static __device__ __noinline__ bool arrive_is_last(uint32_t* counter, uint32_t epoch, int nc, volatile int* abort,
                                            const GemmParams& p, int detail) {
    const uint32_t tag = epoch & 0xFFFFFFu;
    uint32_t old = atomicAdd(counter, 0u);
    for (int tries = 0; tries < (1 << 20); ++tries) {
        const uint32_t count = ((old >> 8) == tag ? (old & 0xFFu) : 0u) + 1u;
        const uint32_t prev = atomicCAS(counter, old, (tag << 8) | count);
        if (prev == old) {
            if (count != (uint32_t)nc) return false;
            atomicExch(counter, 0u);   // every contributor is in: the word is free again
            return true;
        }
        old = prev;
    }
    *abort = 1;
    report_timeout(p, kSiteStreamK, detail);
    return false;
}

// Stage one operand tile of `rows` (M or N) x kBK (K).
template <bool kPair>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, int mn_major,
                                             int row0, int rows, int k0, uint32_t bar, uint64_t policy) {
    if (mn_major) {
        for (int j = 0; j < rows / 64; ++j) {
            if constexpr (kPair)
                ptx::tma_load_2d_pair_hint(dst + j * kMnChunkBytes, map, row0 + 64 * j, k0, bar, policy);
            else
                ptx::tma_load_2d_hint(dst + j * kMnChunkBytes, map, row0 + 64 * j, k0, bar, policy);
        }
    } else {
        if constexpr (kPair)
            ptx::tma_load_2d_pair_hint(dst, map, k0, row0, bar, policy);
        else
            ptx::tma_load_2d_hint(dst, map, k0, row0, bar, policy);
    }
}

// One pipeline stage (kSub K sub-blocks) of an operand.  For stages below
// `whole`, box_dims 3: a K-major operand whose stage map is {K in a 128-byte
// row, rows, K chunks}: one box of all kSub chunks, whose shared image is
// the kSub sub-blocks one after another; box_dims 4: an MN-major operand
// whose stage map is {MN in a 128-byte row, K rows of a chunk, MN chunks,
// K chunks}: one box, laid out as [sub-block][64-wide MN chunk][K row], the
// same image as the 2-D boxes.  Otherwise one 2-D box of `map` per
// sub-block (and per MN chunk).
template <bool kPair, int kSub>
__device__ __forceinline__ void load_stage(uint32_t dst, uint32_t sub_bytes, const CUtensorMap* map,
                                           const CUtensorMap* stage_map, int mn_major, int box_dims, int whole,
                                           int row0, int rows, int kb, int bke, uint32_t bar, uint64_t policy) {
    // The launch-wide 2-D test comes first: testing the stage index inside
    // every branch cost the one-sub-block kernels 22 % at K = 256 (measured).
    if (box_dims != 2 && kb < whole) {
        if (box_dims == 3) {
            if constexpr (kPair)
                ptx::tma_load_3d_pair_hint(dst, stage_map, 0, row0, kb * kSub, bar, policy);
            else
                ptx::tma_load_3d_hint(dst, stage_map, 0, row0, kb * kSub, bar, policy);
        } else {
            if constexpr (kPair)
                ptx::tma_load_4d_pair_hint(dst, stage_map, 0, 0, row0 / 64, kb * kSub, bar, policy);
            else
                ptx::tma_load_4d_hint(dst, stage_map, 0, 0, row0 / 64, kb * kSub, bar, policy);
        }
    } else {
#pragma unroll
        for (int sub = 0; sub < kSub; ++sub)
            load_operand<kPair>(dst + sub * sub_bytes, map, mn_major, row0, rows, (kb * kSub + sub) * bke, bar, policy);
    }
}

template <int kOut>
struct OutTraits;
template <>
struct OutTraits<kOutF32> {
    static constexpr int kBytes = 4;
};
template <>
struct OutTraits<kOutF16> {
    static constexpr int kBytes = 2;
};
template <>
struct OutTraits<kOutBF16> {
    static constexpr int kBytes = 2;
};

__device__ __forceinline__ uint32_t pack2(float a, float b, int out) {
    if (out == kOutF16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack2(uint32_t u, int out) {
    if (out == kOutF16) {
        __half2 h = *reinterpret_cast<__half2*>(&u);
        return __half22float2(h);
    }
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
}

template <bool kPair, int kOut, int kEpiW, bool kHasC, int kTileN, bool kF8, bool kMX = false>
__global__ void __launch_bounds__(Cfg<kPair, kEpiW, kTileN, kMX>::kNumThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmAs, const __grid_constant__ CUtensorMap tmBs,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                        const GemmParams p) {
    using Cf = Cfg<kPair, kEpiW, kTileN, kMX>;
    static_assert(!kMX || kF8, "block scaling applies to 8-bit operands");
    constexpr int kBN = kTileN;
    // K elements per 128-byte operand row; an MMA's K slice is 32 bytes of
    // it either way, so descriptors advance alike (8-bit operands are only
    // ever staged K-major).
    constexpr int kBKe = kF8 ? kBK8 : kBK;
    constexpr int kCG = Cf::kCtaGroup;
    constexpr int kEpiWarps = Cf::kEpiWarps;
    constexpr int kOutBytes = OutTraits<kOut>::kBytes;
    constexpr int kChunkCols = 128 / kOutBytes;   // columns per 128-byte staging row
    constexpr int kChunks = Cf::kEpiCols / kChunkCols;   // staging chunks per warp and tile

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128B-swizzle atoms need 1024-B alignment
    uint8_t* smem = smem_raw + (base - raw);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = kPair ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;

    const uint32_t bars = base + Cf::kOffBar;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (Cf::kStages + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * Cf::kStages + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * Cf::kStages + 2 + a); };
    auto c_bar = [&](int w, int b) { return bars + 8u * (2 * Cf::kStages + 4 + Cf::kEpiBufs * w + b); };
    auto sf_bar = [&](int s) { return bars + 8u * (2 * Cf::kStages + 4 + Cf::kEpiBufs * kEpiWarps + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cf::kOffAbort);
    volatile int* sk_flag = reinterpret_cast<volatile int*>(smem + Cf::kOffSkFlag);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + Cf::kOffTmemSlot);

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cf::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull_bar(a), 1);
            ptx::mbar_init(tempty_bar(a), (kPair ? 2 : 1) * kEpiWarps * 32);
        }
        for (int w = 0; w < kEpiWarps; ++w)
            for (int b = 0; b < Cf::kEpiBufs; ++b) ptx::mbar_init(c_bar(w, b), 1);
        if constexpr (kMX)
            for (int s = 0; s < Cf::kStages; ++s) ptx::mbar_init(sf_bar(s), 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
        // the maps the producer reads: the whole-stage ones first, the 2-D
        // ones where some stage takes them
        if (p.a_box_dims > 2) ptx::prefetch_tensormap(&tmAs);
        if (p.b_box_dims > 2) ptx::prefetch_tensormap(&tmBs);
        if (p.a_box_dims == 2 || p.a_whole_stages < p.num_k_blocks) ptx::prefetch_tensormap(&tmA);
        if (p.b_box_dims == 2 || p.b_whole_stages < p.num_k_blocks) ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmD);
        if constexpr (kHasC) ptx::prefetch_tensormap(&tmC);
        if constexpr (kMX) {
            ptx::prefetch_tensormap(&tmSFA);
            ptx::prefetch_tensormap(&tmSFB);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc<kCG>(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
        ptx::tmem_relinquish<kCG>();
    }
    ptx::tc_fence_before_sync();
    if constexpr (kPair)
        ptx::cluster_sync();
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Launched with programmatic stream serialisation, this grid may start
    // while the previous kernel on the stream is still finishing: the set-up
    // above (barriers, tensor memory, descriptor prefetch) overlaps its tail,
    // and every global access below waits for its completion here.  The next
    // grid may be scheduled right away; it can occupy an SM only once this
    // grid's CTA there has exited, and it waits for this grid in turn.
    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    const int cluster_id = kPair ? blockIdx.x / 2 : blockIdx.x;
    const int num_clusters = kPair ? gridDim.x / 2 : gridDim.x;
    const Schedule sched{p.num_tiles, p.num_k_blocks, num_clusters, p.sk_tiles};

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t stage_tx =
                (kPair ? 2 : 1) * ((kMX && p.operands_packed4 ? Cf::kStageBytes / 2 : Cf::kStageBytes) + Cf::kSfBytes);
            const uint64_t pol_a = ptx::l2_policy(p.hint_a);
            const uint64_t pol_b = ptx::l2_policy(p.hint_b);
            const uint64_t pol_sf = ptx::l2_policy(2);   // scales: re-read by every tile of their row / column
            UnitIter units;
            units.start(sched, cluster_id);
            WorkUnit u;
            bool first_unit = true;
            while (ok && units.next(sched, cluster_id, &u)) {
                const int t = u.tile;
                int mb, nb;
                tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, &mb, &nb);
                const int a_row0 = mb * Cf::kTileM + (int)rank * kBM;
                const int b_row0 = nb * kBN + (int)rank * Cf::kLoadN;
                for (int kb = u.kb; kb < u.ke; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p, kSiteProducerEmpty, t)) {
                        ok = false;
                        break;
                    }
                    const bool skip = p.skip_first_stage && first_unit && kb == u.kb;
                    if (!skip) {
                        const uint32_t fb = kPair ? ptx::map_to_rank(full_bar(stage), 0) : full_bar(stage);
                        if (leader) ptx::mbar_arrive_expect_tx(full_bar(stage), stage_tx);
                        load_stage<kPair, Cf::kSub>(base + Cf::kOffA + stage * Cf::kABytes, Cf::kASubBytes, &tmA,
                                                    &tmAs, p.a_mn_major, p.a_box_dims, p.a_whole_stages, a_row0,
                                                    kBM, kb, kBKe, fb, pol_a);
                        load_stage<kPair, Cf::kSub>(base + Cf::kOffB + stage * Cf::kBBytes, Cf::kBSubBytes, &tmB,
                                                    &tmBs, p.b_mn_major, p.b_box_dims, p.b_whole_stages, b_row0,
                                                    Cf::kLoadN, kb, kBKe, fb, pol_b);
                        if constexpr (kMX) {
                            // this stage's scales, laid out by the host in the
                            // order tcgen05.cp reads them (512-byte chunks, rows
                            // of the SFA / SFB tensor maps): per sub-block the
                            // CTA's 128 rows of A, then every column of the tile
#pragma unroll
                            for (int sub = 0; sub < Cf::kSub; ++sub) {
                                const int kc = kb * Cf::kSub + sub;   // 128-K chunk
                                const uint32_t sdst = base + Cf::kOffSf + stage * Cf::kSfBytes + sub * Cf::kSfSubBytes;
                                const int a_chunk = kc * p.sf_a_groups + mb * (kPair ? 2 : 1) + (int)rank;
                                const int b_chunk = (kc * p.num_n_tiles + nb) * Cf::kSfbChunks;
                                if constexpr (kPair) {
                                    ptx::tma_load_2d_pair_hint(sdst, &tmSFA, 0, a_chunk, fb, pol_sf);
                                    ptx::tma_load_2d_pair_hint(sdst + kSfChunkBytes, &tmSFB, 0, b_chunk, fb, pol_sf);
                                } else {
                                    ptx::tma_load_2d_hint(sdst, &tmSFA, 0, a_chunk, fb, pol_sf);
                                    ptx::tma_load_2d_hint(sdst + kSfChunkBytes, &tmSFB, 0, b_chunk, fb, pol_sf);
                                }
                            }
                        }
                    }
                    if (++stage == Cf::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                first_unit = false;
            }
            // Drain: wait until the MMA has released every stage, so that no
            // completion signal is still on its way to this CTA at exit.
            for (int i = 0; ok && i < Cf::kStages; ++i) {
                if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p, kSiteProducerTail, i)) break;
                if (++stage == Cf::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (the pair's leader CTA only) ----------------
        if (leader && lane == 0) {
            const uint32_t idesc = p.idesc;
            // Descriptors of stage 0, K slice 0.  A stage or a K slice moves
            // only the 14-bit start-address field (address >> 4), which cannot
            // carry out of its field: shared addresses stay below 256 KiB.  So
            // the loop advances them with plain adds; this single thread must
            // issue a stage's four MMAs faster than the tensor core runs them.
            const uint64_t a_desc0 = operand_desc(base + Cf::kOffA, p.a_mn_major, 0);
            const uint64_t b_desc0 = operand_desc(base + Cf::kOffB, p.b_mn_major, 0);
            const uint64_t a_kstep = (uint64_t)((p.a_mn_major ? kUK * 128 : kUK * 2) >> 4);
            const uint64_t b_kstep = (uint64_t)((p.b_mn_major ? kUK * 128 : kUK * 2) >> 4);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t gstage = 0;   // stages consumed so far (kMX: picks the scale slot)
            int it = 0;
            bool ok = true;
            UnitIter units;
            units.start(sched, cluster_id);
            WorkUnit u;
            for (; ok && units.next(sched, cluster_id, &u); ++it) {
                const int t = u.tile;
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_bounded(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p, kSiteMmaTmemEmpty, t)) break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
                for (int kb = u.kb; kb < u.ke; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, p, kSiteMmaFull, t)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t ad = a_desc0 + (uint64_t)(stage * (Cf::kABytes >> 4));
                    const uint64_t bd = b_desc0 + (uint64_t)(stage * (Cf::kBBytes >> 4));
                    if constexpr (kMX) {
                        // The scale warp has copied the stage's scales into the
                        // stage's TMEM slot behind the accumulators (16 columns
                        // per sub-block) and committed that to scales_ready;
                        // slice kk of a sub-block takes byte kk of every row's
                        // and column's scale word.
                        if (!wait_bounded(sf_bar(stage), phase, abort_flag, p, kSiteMmaFull, t)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        const uint32_t slot0 =
                            tmem_base + (uint32_t)(2 * kBN + (int)(gstage % Cf::kSfSlots) * Cf::kSfStageCols);
#pragma unroll
                        for (int sub = 0; sub < Cf::kSub; ++sub) {
                            const uint64_t as = ad + (uint64_t)(sub * (Cf::kASubBytes >> 4));
                            const uint64_t bs = bd + (uint64_t)(sub * (Cf::kBSubBytes >> 4));
                            const uint32_t slot = slot0 + sub * kSfSlotCols;
#pragma unroll
                            for (int kk = 0; kk < kBK / kUK; ++kk) {
                                const uint32_t accumulate = ((kb - u.kb) | sub | kk) != 0;
                                ptx::mma_mxf8f6f4<kCG>(d_tmem, as + kk * a_kstep, bs + kk * b_kstep,
                                                       idesc | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), slot,
                                                       slot + 4, accumulate);
                            }
                        }
                    } else {
#pragma unroll
                        for (int sub = 0; sub < Cf::kSub; ++sub) {
                            const uint64_t as = ad + (uint64_t)(sub * (Cf::kASubBytes >> 4));
                            const uint64_t bs = bd + (uint64_t)(sub * (Cf::kBSubBytes >> 4));
#pragma unroll
                            for (int kk = 0; kk < kBK / kUK; ++kk) {
                                const uint32_t accumulate = ((kb - u.kb) | sub | kk) != 0;
                                if constexpr (kF8)
                                    ptx::mma_f8f6f4<kCG>(d_tmem, as + kk * a_kstep, bs + kk * b_kstep, idesc,
                                                         accumulate);
                                else
                                    ptx::mma_f16<kCG>(d_tmem, as + kk * a_kstep, bs + kk * b_kstep, idesc, accumulate);
                            }
                        }
                    }
                    if constexpr (kPair)
                        ptx::mma_commit_pair(empty_bar(stage), 0x3);
                    else
                        ptx::mma_commit(empty_bar(stage));
                    ++gstage;
                    if (++stage == Cf::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (kPair)
                    ptx::mma_commit_pair(tfull_bar(acc), 0x3);
                else
                    ptx::mma_commit(tfull_bar(acc));
            }
        }
        __syncwarp();
    } else if (warp == 2 + kEpiWarps) {
        // ---------------- kMX: scale copies (the pair's leader CTA only) ----------------
        // For each stage the MMA issuer will use, in the same order: wait for
        // its data, copy its scales from shared memory into a TMEM scale slot
        // (slot g mod kSfSlots for the g-th stage; tcgen05.cp, in both CTAs of
        // a pair), commit to scales_ready.  Taking the copies off the MMA
        // issuer shortens its per-stage work.  The slot's previous readers,
        // the MMAs of stage g - kSfSlots, have completed: with one slot per
        // stage, because the producer refilled this stage only after their
        // commit released it and the full barrier waited on here follows that
        // refill; with fewer slots than stages, by waiting for that commit on
        // its stage's empty barrier (whose next phase cannot complete before
        // this warp has copied stage g + 1, so the parity test is unambiguous).
        if constexpr (kMX) {
            if (leader && lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t gstage = 0;
                bool ok = true;
                UnitIter units;
                units.start(sched, cluster_id);
                WorkUnit u;
                while (ok && units.next(sched, cluster_id, &u)) {
                    for (int kb = u.kb; kb < u.ke; ++kb) {
                        if (!wait_bounded(full_bar(stage), phase, abort_flag, p, kSiteMmaFull, u.tile)) {
                            ok = false;
                            break;
                        }
                        if constexpr (Cf::kSfSlots < Cf::kStages) {
                            if (gstage >= (uint32_t)Cf::kSfSlots) {
                                const uint32_t prev = gstage - Cf::kSfSlots;
                                if (!wait_bounded(empty_bar((int)(prev % Cf::kStages)), (prev / Cf::kStages) & 1u,
                                                  abort_flag, p, kSiteMmaFull, u.tile)) {
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        ptx::tc_fence_after_sync();
                        const uint32_t slot0 =
                            tmem_base + (uint32_t)(2 * kBN + (int)(gstage % Cf::kSfSlots) * Cf::kSfStageCols);
                        const uint32_t ssrc0 = base + Cf::kOffSf + stage * Cf::kSfBytes;
#pragma unroll
                        for (int sub = 0; sub < Cf::kSub; ++sub) {
                            const uint32_t slot = slot0 + sub * kSfSlotCols;
                            const uint32_t ssrc = ssrc0 + sub * Cf::kSfSubBytes;
                            ptx::tmem_cp_32x128b_warpx4<kCG>(slot, sf_desc(ssrc));
#pragma unroll
                            for (int c = 0; c < Cf::kSfbChunks; ++c)
                                ptx::tmem_cp_32x128b_warpx4<kCG>(slot + 4 + 4 * c,
                                                                 sf_desc(ssrc + (1 + c) * kSfChunkBytes));
                        }
                        if constexpr (kPair)
                            ptx::mma_commit_pair(sf_bar(stage), 0x1);
                        else
                            ptx::mma_commit(sf_bar(stage));
                        ++gstage;
                        if (++stage == Cf::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 2 .. 2 + kEpiW - 1 ----------------
        const int ew = warp - 2;   // staging buffers and C barriers of this warp
        const int q = warp & 3;    // the TMEM lane quadrant this warp may read
        const int col_begin = (ew / 4) * Cf::kEpiCols;   // this warp's first column in the tile
        const uint32_t epi = base + Cf::kOffEpi + ew * Cf::kEpiBufs * kEpiBufBytes;
        const float alpha = p.alpha;
        const float beta = p.beta;
        constexpr int kVec = 16 / kOutBytes;   // elements per 16-byte piece
        const uint64_t pol_d = ptx::l2_policy(p.hint_d);
        // C is read exactly once: evict-first, so that it does not push the
        // operand panels the other tiles still read out of L2 (4096^3 E5M2
        // beta = 1: +1.8 %, bf16: +0.3 %).
        const uint64_t pol_c = ptx::l2_policy(1);
        uint32_t chunk_iter = 0;
        int it = 0;
        bool ok = true;
        UnitIter units;
        units.start(sched, cluster_id);
        WorkUnit u;
        for (; ok && units.next(sched, cluster_id, &u); ++it) {
            const int t = u.tile;
            int mb, nb;
            tile_coords(t, p.num_m_tiles, p.num_n_tiles, p.group_m, &mb, &nb);
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            const int row0 = mb * Cf::kTileM + (int)rank * kBM + q * 32;
            // C does not depend on the main loop: for a whole tile, the C
            // boxes of the first kEpiBufs chunks are fetched before the
            // accumulator is ready, so their latency hides behind the MMAs.
            // (A stream-K contributor learns only later whether it stores.)
            constexpr int kPrefetchC = kHasC ? (Cf::kEpiBufs < kChunks ? Cf::kEpiBufs : kChunks) : 0;
            const bool prefetch_c = kPrefetchC > 0 && u.nc == 1;
            if (prefetch_c && lane == 0) {
                ptx::bulk_wait_group_read<0>();   // every staging box of this warp is free
#pragma unroll
                for (int c = 0; c < kPrefetchC; ++c) {
                    const int col0 = nb * kBN + col_begin + c * kChunkCols;
                    if (col0 < p.N) {
                        const uint32_t buf = (chunk_iter + c) % Cf::kEpiBufs;
                        ptx::mbar_arrive_expect_tx(c_bar(ew, buf), kEpiBufBytes);
                        ptx::tma_load_2d_hint(epi + buf * kEpiBufBytes, &tmC, col0, row0, c_bar(ew, buf), pol_c);
                    }
                }
            }
            ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag, p, kSiteEpilogueTmemFull, t);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after_sync();
            const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN + col_begin);
            bool more = false;
            if (p.epi_pace_ns > 0) {
                UnitIter peek = units;
                WorkUnit nu;
                more = peek.next(sched, cluster_id, &nu);
            }
            const bool pace = more;

            // Stream-K: a unit that covers only part of its tile's K range
            // stores its partial accumulator, then counts itself in; only the
            // last contributor to arrive goes on to finish the tile (adding
            // every contributor's partial in contributor order, so the result
            // does not depend on who arrives last).
            const bool partial = u.nc > 1;
            const float4* ws = static_cast<const float4*>(p.ws_partials);
            auto partial_at = [&](int contributor, int unit32, int j) -> int64_t {
                const int64_t slot = (int64_t)u.sk * p.ws_max_nc + contributor;
                return (slot * 2 + rank) * (kBM * kBN / 4) + ((q * (kBN / 32) + unit32) * 8 + j) * 32 + lane;
            };
            if (partial) {
                __syncwarp();
#pragma unroll 1
                for (int g = 0; g < Cf::kEpiCols / 32; ++g) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(g * 32), r);
                    ptx::tmem_wait_ld(r);
                    float4* dst = static_cast<float4*>(p.ws_partials);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(&dst[partial_at(u.ci, col_begin / 32 + g, j)],
                               make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                           __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
                }
                __threadfence();
                epi_bar_sync<kEpiWarps>();
                if (ew == 0 && lane == 0)
                    *sk_flag = arrive_is_last(p.ws_counters + (u.sk * 2 + rank), p.ws_epoch, u.nc, abort_flag, p, t)
                                   ? 1
                                   : 0;
                epi_bar_sync<kEpiWarps>();
                const bool last = *sk_flag != 0;
                if (!last) {
                    ptx::tc_fence_before_sync();
                    if constexpr (kPair)
                        ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
                    else
                        ptx::mbar_arrive(tempty_bar(acc));
                    continue;
                }
                __threadfence();
                // Last to arrive: replace this CTA's accumulator in TMEM by the
                // sum of every contributor's partial, in contributor order (its
                // own term read back from TMEM), then finish the tile as usual.
                __syncwarp();   // the tcgen05 loads / stores below are .sync.aligned
#pragma unroll 1
                for (int g = 0; g < Cf::kEpiCols / 32; ++g) {
                    uint32_t r[32];
                    ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(g * 32), r);
                    ptx::tmem_wait_ld(r);
                    const int unit32 = col_begin / 32 + g;
                    float4 s[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) s[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int k = 0; k < u.nc; ++k) {
                        float4 x[8];
                        if (k == u.ci) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                x[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                        } else {
                            // the eight loads are independent: all in flight together
#pragma unroll
                            for (int j = 0; j < 8; ++j) x[j] = __ldcg(&ws[partial_at(k, unit32, j)]);
                        }
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            s[j].x += x[j].x;
                            s[j].y += x[j].y;
                            s[j].z += x[j].z;
                            s[j].w += x[j].w;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        r[4 * j] = __float_as_uint(s[j].x);
                        r[4 * j + 1] = __float_as_uint(s[j].y);
                        r[4 * j + 2] = __float_as_uint(s[j].z);
                        r[4 * j + 3] = __float_as_uint(s[j].w);
                    }
                    ptx::tmem_st_32x32b_x32(t_row + (uint32_t)(g * 32), r);
                }
                ptx::tmem_wait_st();
            }
            // Accumulator chunks come out of TMEM one ahead of their use: the
            // load of chunk c+1 is in flight while chunk c is converted and
            // staged.  Two named register arrays alternate (chunks are taken
            // in pairs), so the asynchronously written registers are never
            // copied or indexed at run time before their wait.
            uint32_t va[kChunkCols], vb[kChunkCols];
            auto tmem_load = [&](int c, uint32_t(&v)[kChunkCols]) {
                ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kChunkCols), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                if constexpr (kChunkCols == 64)
                    ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(c * kChunkCols + 32),
                                            *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            };
            bool stop = false;
            auto chunk = [&](int c, uint32_t(&v)[kChunkCols], uint32_t(&next)[kChunkCols]) {
                if (stop) return;
                // tcgen05.ld / wait::ld are .sync.aligned: the previous chunk
                // ended in lane-dependent code (the ragged-column stores), so
                // the warp reconverges explicitly first.
                __syncwarp();
                ptx::tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                if constexpr (kChunkCols == 64) ptx::tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                const uint32_t buf = chunk_iter % Cf::kEpiBufs;
                const uint32_t sbuf = epi + buf * kEpiBufBytes;
                const int col0 = nb * kBN + col_begin + c * kChunkCols;
                if (col0 >= p.N) {   // the rest of this tile lies beyond the last column
                    stop = true;
                    return;
                }
                if (c + 1 < kChunks) tmem_load(c + 1, next);
                // Every chunk commits one bulk group (empty when it stores
                // nothing), so allowing kEpiBufs - 1 groups in flight means the
                // store that last used this buffer has finished reading it.
                if (lane == 0) ptx::bulk_wait_group_read<Cf::kEpiBufs - 1>();
                __syncwarp();
                if constexpr (kHasC) {   // this chunk of C, by TMA, into the staging box
                    // C runs kAhead chunks ahead of its use: chunk c's C was
                    // prefetched with the tile or issued by chunk c - kAhead;
                    // only the first chunks of a tile without the prefetch
                    // load their own.  Then this chunk issues the C of chunk
                    // c + kAhead into the buffer of chunk c - 1, once that
                    // chunk's D store has read it, so the load's latency hides
                    // behind this chunk's work.
                    constexpr int kAhead = Cf::kEpiBufs - 1;
                    if (lane == 0 && !((prefetch_c && c < kPrefetchC) || c >= kAhead)) {
                        ptx::mbar_arrive_expect_tx(c_bar(ew, buf), kEpiBufBytes);
                        ptx::tma_load_2d_hint(sbuf, &tmC, col0, row0, c_bar(ew, buf), pol_c);
                    }
                    const int cn = c + kAhead;
                    if (kAhead > 0 && cn < kChunks && !(prefetch_c && cn < kPrefetchC) &&
                        col0 + kAhead * kChunkCols < p.N && lane == 0) {
                        ptx::bulk_wait_group_read<0>();
                        const uint32_t bn = (chunk_iter + kAhead) % Cf::kEpiBufs;
                        ptx::mbar_arrive_expect_tx(c_bar(ew, bn), kEpiBufBytes);
                        ptx::tma_load_2d_hint(epi + bn * kEpiBufBytes, &tmC, col0 + kAhead * kChunkCols, row0,
                                         c_bar(ew, bn), pol_c);
                    }
                    ok = wait_bounded(c_bar(ew, buf), (chunk_iter / Cf::kEpiBufs) & 1u, abort_flag, p,
                                      kSiteEpilogueC, t);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) {
                        stop = true;
                        return;
                    }
                }
                const uint32_t row_addr = sbuf + (uint32_t)lane * 128u;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t addr = row_addr + ((uint32_t)(j ^ (lane & 7)) << 4);
                    uint32_t w[4];
                    if constexpr (kOutBytes == 4) {
                        float o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[e] = alpha * __uint_as_float(v[4 * j + e]);
                        if constexpr (kHasC) {
                            uint32_t c4[4];
                            ptx::ld_shared_v4(addr, c4[0], c4[1], c4[2], c4[3]);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = fmaf(alpha, __uint_as_float(v[4 * j + e]), beta * __uint_as_float(c4[e]));
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(o[e]);
                    } else {
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = alpha * __uint_as_float(v[8 * j + e]);
                        if constexpr (kHasC) {
                            uint32_t c4[4];
                            ptx::ld_shared_v4(addr, c4[0], c4[1], c4[2], c4[3]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 cf = unpack2(c4[e], kOut);
                                o[2 * e] = fmaf(alpha, __uint_as_float(v[8 * j + 2 * e]), beta * cf.x);
                                o[2 * e + 1] = fmaf(alpha, __uint_as_float(v[8 * j + 2 * e + 1]), beta * cf.y);
                            }
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) w[e] = pack2(o[2 * e], o[2 * e + 1], kOut);
                    }
                    ptx::st_shared_v4(addr, w[0], w[1], w[2], w[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                const bool tma_part = col0 < p.n_tma;
                if (lane == 0) {
                    if (tma_part) ptx::tma_store_2d_hint(&tmD, sbuf, col0, row0, pol_d);
                    ptx::bulk_commit_group();
                }
                // columns [n_tma, N) of this row, one element at a time
                if (col0 + kChunkCols > p.n_tma && row0 + lane < p.M) {
                    const int c_begin = col0 > p.n_tma ? col0 : p.n_tma;
                    const int c_end = col0 + kChunkCols < p.N ? col0 + kChunkCols : p.N;
                    char* drow = static_cast<char*>(p.d_ptr) + ((int64_t)(row0 + lane) * p.ldd) * kOutBytes;
                    for (int col = c_begin; col < c_end; ++col) {
                        const int cc = col - col0;
                        const uint32_t addr =
                            row_addr + ((uint32_t)((cc / kVec) ^ (lane & 7)) << 4) + (uint32_t)((cc % kVec) * kOutBytes);
                        if constexpr (kOutBytes == 4)
                            *reinterpret_cast<uint32_t*>(drow + (int64_t)col * 4) = ptx::ld_shared_u32(addr);
                        else
                            *reinterpret_cast<uint16_t*>(drow + (int64_t)col * 2) = ptx::ld_shared_u16(addr);
                    }
                }
                if (pace) __nanosleep((unsigned)p.epi_pace_ns);
                ++chunk_iter;
            };
            static_assert(kChunks >= 1, "at least one staging chunk per warp and tile");
            __syncwarp();
            tmem_load(0, va);
#pragma unroll
            for (int c = 0; c < kChunks; c += 2) {
                chunk(c, va, vb);
                if (c + 1 < kChunks) chunk(c + 1, vb, va);
            }
            __syncwarp();
            ptx::tmem_wait_ld();   // a prefetch cut short by `stop` must land before the release
            if (!ok) break;
            // every TMEM read of this accumulator has completed (wait::ld)
            ptx::tc_fence_before_sync();
            if constexpr (kPair)
                ptx::mbar_arrive_cluster(ptx::map_to_rank(tempty_bar(acc), 0));
            else
                ptx::mbar_arrive(tempty_bar(acc));
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    if constexpr (kPair)
        ptx::cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc<kCG>(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host-side launch helpers (templates; instantiated by the including unit)

// Instantiated configurations: every (pair, beta != 0) combination of the
// 256-wide tiles with 4 epilogue warps for each output type, and with 8
// epilogue warps for f32 output (the store-bound configuration); the
// 224-wide CTA-pair tiles with 4 epilogue warps for f32 output; the 64-wide
// single-CTA tiles with 4 epilogue warps for each output type.
template <bool kPair, int kOut, int kEpiW, bool kHasC, int kTileN, bool kF8, bool kMX = false>
static cudaError_t prepare_one() {
    return cudaFuncSetAttribute(gemm_tcgen05_kernel<kPair, kOut, kEpiW, kHasC, kTileN, kF8, kMX>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<kPair, kEpiW, kTileN, kMX>::kSmemBytes);
}

template <bool kPair, bool kHasC, bool kF8>
static cudaError_t prepare_group() {
    cudaError_t e;
    if ((e = prepare_one<kPair, kOutF32, 4, kHasC, kBNMax, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_one<kPair, kOutF32, 8, kHasC, kBNMax, kF8>()) != cudaSuccess) return e;
    if constexpr (kPair)
        if ((e = prepare_one<kPair, kOutF32, 4, kHasC, kFitN, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_one<kPair, kOutF16, 4, kHasC, kBNMax, kF8>()) != cudaSuccess) return e;
    return prepare_one<kPair, kOutBF16, 4, kHasC, kBNMax, kF8>();
}

template <bool kHasC, bool kF8>
static cudaError_t prepare_narrow() {
    cudaError_t e;
    if ((e = prepare_one<false, kOutF32, 4, kHasC, kNarrowN, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_one<false, kOutF16, 4, kHasC, kNarrowN, kF8>()) != cudaSuccess) return e;
    return prepare_one<false, kOutBF16, 4, kHasC, kNarrowN, kF8>();
}

template <bool kPair, int kOut, int kEpiW, bool kHasC, int kTileN, bool kF8, bool kMX = false>
static cudaError_t launch_one(const TcgenLaunch& L, cudaStream_t stream) {
    using Cf = Cfg<kPair, kEpiW, kTileN, kMX>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid, 1, 1);
    cfg.blockDim = dim3(Cf::kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (kPair) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (L.pdl) {   // programmatic dependent launch (see grid_dependency_wait in the kernel)
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<kPair, kOut, kEpiW, kHasC, kTileN, kF8, kMX>, L.a, L.b,
                              L.a_stage, L.b_stage, L.c, L.d, L.sfa, L.sfb, L.p);
}

template <bool kPair, bool kHasC, bool kF8>
static cudaError_t launch_group(const TcgenLaunch& L, cudaStream_t stream) {
    if (L.tile_n == kFitN) {   // f32 D, 4 epilogue warps, CTA pairs (the host's plan guarantees it)
        if constexpr (kPair)
            if (L.out == kOutF32 && L.epi_warps == 4) return launch_one<kPair, kOutF32, 4, kHasC, kFitN, kF8>(L, stream);
        return cudaErrorInvalidConfiguration;
    }
    if (L.out == kOutF32)
        return L.epi_warps == 8 ? launch_one<kPair, kOutF32, 8, kHasC, kBNMax, kF8>(L, stream)
                                : launch_one<kPair, kOutF32, 4, kHasC, kBNMax, kF8>(L, stream);
    if (L.out == kOutF16) return launch_one<kPair, kOutF16, 4, kHasC, kBNMax, kF8>(L, stream);
    return launch_one<kPair, kOutBF16, 4, kHasC, kBNMax, kF8>(L, stream);
}

template <bool kHasC, bool kF8>
static cudaError_t launch_narrow(const TcgenLaunch& L, cudaStream_t stream) {
    if (L.out == kOutF32) return launch_one<false, kOutF32, 4, kHasC, kNarrowN, kF8>(L, stream);
    if (L.out == kOutF16) return launch_one<false, kOutF16, 4, kHasC, kNarrowN, kF8>(L, stream);
    return launch_one<false, kOutBF16, 4, kHasC, kNarrowN, kF8>(L, stream);
}


// Every configuration of one operand family (kF8: E4M3 / E5M2, else fp16 /
// bf16): its shared-memory limits, and the launch that dispatches on L.
template <bool kF8>
static cudaError_t prepare_family() {
    cudaError_t e;
    if ((e = prepare_group<false, false, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_group<false, true, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_group<true, false, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_group<true, true, kF8>()) != cudaSuccess) return e;
    if ((e = prepare_narrow<false, kF8>()) != cudaSuccess) return e;
    return prepare_narrow<true, kF8>();
}

template <bool kF8>
static cudaError_t launch_family(const TcgenLaunch& L, cudaStream_t stream) {
    const bool has_c = L.p.has_c != 0;
    if (L.tile_n == kNarrowN)
        return has_c ? launch_narrow<true, kF8>(L, stream) : launch_narrow<false, kF8>(L, stream);
    if (L.pair) return has_c ? launch_group<true, true, kF8>(L, stream) : launch_group<true, false, kF8>(L, stream);
    return has_c ? launch_group<false, true, kF8>(L, stream) : launch_group<false, false, kF8>(L, stream);
}

// The block-scaled kernels: 224-wide (f32 D) or 192-wide (16-bit D) tiles on
// one SM or a CTA pair, 4 epilogue warps, with and without C.
template <bool kPair, bool kHasC>
static cudaError_t prepare_mx_group() {
    cudaError_t e;
    if ((e = prepare_one<kPair, kOutF32, 4, kHasC, kMxTileNF32, true, true>()) != cudaSuccess) return e;
    if ((e = prepare_one<kPair, kOutF16, 4, kHasC, kMxTileN, true, true>()) != cudaSuccess) return e;
    return prepare_one<kPair, kOutBF16, 4, kHasC, kMxTileN, true, true>();
}

template <bool kPair, bool kHasC>
static cudaError_t launch_mx_group(const TcgenLaunch& L, cudaStream_t stream) {
    if (L.out == kOutF32) return launch_one<kPair, kOutF32, 4, kHasC, kMxTileNF32, true, true>(L, stream);
    if (L.out == kOutF16) return launch_one<kPair, kOutF16, 4, kHasC, kMxTileN, true, true>(L, stream);
    return launch_one<kPair, kOutBF16, 4, kHasC, kMxTileN, true, true>(L, stream);
}

}  // namespace gb300
