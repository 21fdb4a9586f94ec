// Internal interface between the C-ABI host code (gemm_api.cpp) and the
// sm_103a kernels (gemm_tcgen05.cuh instantiated by gemm_sm103.cu and
// gemm_sm103_f8.cu and gemm_sm103_mx.cu; gemm_mma_sync.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_params.h"

namespace gb300 {

// Output (C and D) element types, in the kernels' template vocabulary.
enum OutKind : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

// Device status code written by a wait that gave up (= GEMM_ERR_DEVICE_TIMEOUT).
constexpr int kDeviceErrTimeout = -8;

struct TcgenLaunch {
    CUtensorMap a, b, c, d;   // TMA descriptors (c unused when beta == 0)
    CUtensorMap sfa, sfb;     // block scales (mx only; see GemmParams::sf_a_groups)
    CUtensorMap a_stage, b_stage;   // whole-stage boxes (see GemmParams::a_box_dims)
    GemmParams p;
    int pair;                 // 1: CTA-pair (cta_group::2) kernel
    int out;                  // OutKind
    int grid;                 // CTAs (a multiple of 2 for the pair kernel)
    int epi_warps;            // 4 or 8 epilogue warps
    int tile_n;               // 256, or 64 for the narrow single-CTA tiles
    int f8;                   // 1: E4M3 / E5M2 operands (kind::f8f6f4), K-major only
    int mx;                   // 1: MX block-scaled (kind::mxf8f6f4; 8-bit or packed E2M1 operands), 192-wide tiles
    int pdl;                  // 1: launch with programmatic stream serialisation
};

// Arguments of the warp-level mma.sync path (gemm_mma_sync.cu): any
// element-aligned layout; K > 0.
struct SyncParams {
    const void* A;
    const void* B;
    const void* C;
    void* D;
    int64_t M, N, K, lda, ldb, ldc, ldd;
    int transA, transB;
    float alpha, beta;
    int in_bf16;   // A and B are bf16 (else f16)
    int out;       // OutKind of C and D
    int has_c;     // beta != 0
    int atom;      // 1: the one-warp-per-16x8-block kernel (tiny problems), 0: the tiled one
};

cudaError_t launch_mma_sync(const SyncParams& p, cudaStream_t stream);

// 1 unless GEMM_PDL=0: launch kernels with programmatic stream serialisation
// (each kernel waits for its predecessor with griddepcontrol.wait before its
// first global access, so its set-up overlaps the predecessor's tail).
int pdl_setting();

#ifdef __CUDACC__
// Launches `kernel` on `stream`, with programmatic stream serialisation
// when pdl_setting() allows it.
template <typename... KArgs, typename... Args>
cudaError_t launch_with_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_setting() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
#endif

// dst[r * ldd + c] = src[r * lds + c] for r < rows, c < cols; elements of
// elem_bytes (1, 2 or 4) bytes, any element-aligned strides.
cudaError_t launch_copy2d(void* dst, int64_t ldd, const void* src, int64_t lds, int64_t rows, int64_t cols,
                          int elem_bytes, cudaStream_t stream);
// dst[c * ldd + r] = src[r * lds + c] (dst holds the cols x rows transpose);
// elements of 1 or 2 bytes.
cudaError_t launch_transpose2d(void* dst, int64_t ldd, const void* src, int64_t lds, int64_t rows, int64_t cols,
                               int elem_bytes, cudaStream_t stream);

cudaError_t prepare_kernels_on_current_device();
cudaError_t launch_tcgen05(const TcgenLaunch& L, cudaStream_t stream);
cudaError_t prepare_kernels_f8();                                          // gemm_sm103_f8.cu
cudaError_t launch_tcgen05_f8(const TcgenLaunch& L, cudaStream_t stream);  // gemm_sm103_f8.cu
cudaError_t prepare_kernels_mx();                                          // gemm_sm103_mx.cu
cudaError_t launch_tcgen05_mx(const TcgenLaunch& L, cudaStream_t stream);  // gemm_sm103_mx.cu
// MX scales of one operand, [rows, kblocks] bytes with row stride ld, into
// the block-scaled kernel's 512-byte chunks (see GemmParams::sf_a_groups)
// for tiles of tile_rows rows (columns) and kchunks 128-K sub-blocks; rows
// and blocks outside the matrix get the scale 1 (byte 127).
// One operand's block scales for sf_tiles_kernel (see gemm_sm103_mx.cu).
struct SfJob {
    uint32_t* out;          // rearranged chunks (sf_tiles_bytes)
    const uint8_t* in;      // the caller's scales, [rows][ld] bytes
    int64_t ld, rows, kblocks;
    int32_t tile_rows, groups;
    int64_t tiles, kchunks;
    int64_t blocks;         // thread blocks of this job
};
SfJob sf_job(uint8_t* out, const uint8_t* in, int64_t ld, int64_t rows, int64_t kblocks, int tile_rows, int64_t tiles,
             int64_t kchunks);
cudaError_t launch_sf_tiles(const SfJob& a, const SfJob& b, cudaStream_t stream);   // both in one launch
int64_t sf_tiles_bytes(int tile_rows, int64_t tiles, int64_t kchunks);
int tcgen05_mx_tile_n(int f32_out);   // D columns per block-scaled tile
int tcgen05_mx_smem_bytes(int pair, int f32_out);
int tcgen05_mx_stages(int pair, int f32_out);
cudaError_t launch_k0(int out, void* D, const void* C, int M, int N, int64_t ldc, int64_t ldd, float alpha,
                      float beta, int has_c, int num_sms, cudaStream_t stream);

// Static scratch of gemm_noalloc(): its device address on the current
// device (cudaGetSymbolAddress) and its size in bytes.
cudaError_t noalloc_scratch_address(void** ptr);
int noalloc_scratch_bytes();

int tcgen05_tile_m(int pair);      // D rows per tile
int tcgen05_wide_n();              // D columns per throughput tile
int tcgen05_narrow_n();            // D columns per narrow tile (single CTA, 4 epilogue warps)
int tcgen05_fit_n();               // D columns per wave-fitted tile (CTA pair, f32 D, K-major B)
int tcgen05_block_k(int f8);       // K of one TMA operand box (one 128-byte swizzle row)
int tcgen05_stage_k(int pair, int f8, int epi_warps, int tile_n);   // K per pipeline stage
int tcgen05_load_rows_a();         // A rows (M) one CTA stages per stage
int tcgen05_load_rows_b(int pair, int tile_n);   // B rows (N) one CTA stages per stage
int tcgen05_smem_bytes(int pair, int epi_warps, int tile_n);
int tcgen05_stages(int pair, int epi_warps, int tile_n);

}  // namespace gb300
