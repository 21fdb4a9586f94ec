// Instantiations of the tcgen05 kernel for fp16 / bf16 operands, the K = 0
// kernel, the allocation-free entry point's static scratch, and the host-side
// queries and launchers gemm_api.cpp calls.  The kernel itself is in
// gemm_tcgen05.cuh; gemm_sm103_f8.cu instantiates it for 8-bit operands.
#include "gemm_tcgen05.cuh"

namespace gb300 {

// K = 0: the sum is empty, D = alpha * 0 + beta * C (C not read when beta = 0).
template <int kOut>
__global__ void gemm_k0_kernel(void* D, const void* C, int M, int N, int64_t ldc, int64_t ldd, float alpha,
                               float beta, int has_c) {
    ptx::grid_dependency_wait();   // the previous kernel's writes are visible (programmatic launch)
    ptx::launch_dependents();
    const int64_t total = (int64_t)M * N;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / N, j = idx - (idx / N) * N;
        const float acc = 0.0f;
        float d = alpha * acc;
        if (kOut == kOutF32) {
            if (has_c) d = fmaf(alpha, acc, beta * static_cast<const float*>(C)[i * ldc + j]);
            static_cast<float*>(D)[i * ldd + j] = d;
        } else if (kOut == kOutF16) {
            if (has_c) d = fmaf(alpha, acc, beta * __half2float(static_cast<const __half*>(C)[i * ldc + j]));
            static_cast<__half*>(D)[i * ldd + j] = __float2half_rn(d);
        } else {
            if (has_c)
                d = fmaf(alpha, acc, beta * __bfloat162float(static_cast<const __nv_bfloat16*>(C)[i * ldc + j]));
            static_cast<__nv_bfloat16*>(D)[i * ldd + j] = __float2bfloat16_rn(d);
        }
    }
}

// ---------------------------------------------------------------------------
// Scratch of the allocation-free entry point gemm_noalloc(): the device
// status record its launches write lives in this fixed module array (zeroed
// when the module loads, kept by every GPU that loads the library until the
// process exits) instead of in a cudaMalloc'd block.  Every gemm_noalloc()
// call on a device shares it.

constexpr int kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static_assert(sizeof(DeviceStatus) <= kNoAllocScratchBytes, "the status record must fit the static scratch");

// Device address of the static scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address must come
// from the runtime; call with the target device current.
cudaError_t noalloc_scratch_address(void** ptr) { return cudaGetSymbolAddress(ptr, g_noalloc_scratch); }

int noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// ---------------------------------------------------------------------------
// host-side launch helpers (called from gemm_api.cpp)

cudaError_t prepare_kernels_on_current_device() {
    cudaError_t e = prepare_family<false>();
    if (e == cudaSuccess) e = prepare_kernels_f8();
    return e != cudaSuccess ? e : prepare_kernels_mx();
}

cudaError_t launch_tcgen05(const TcgenLaunch& L, cudaStream_t stream) {
    if (L.mx) return launch_tcgen05_mx(L, stream);
    return L.f8 ? launch_tcgen05_f8(L, stream) : launch_family<false>(L, stream);
}

int tcgen05_tile_m(int pair) { return pair ? Cfg<true, 4>::kTileM : Cfg<false, 4>::kTileM; }
int tcgen05_wide_n() { return kBNMax; }
int tcgen05_narrow_n() { return kNarrowN; }
int tcgen05_fit_n() { return kFitN; }
int tcgen05_block_k(int f8) { return f8 ? kBK8 : kBK; }
int tcgen05_stage_k(int pair, int f8, int epi_warps, int tile_n) {
    if (tile_n == kNarrowN) return tcgen05_block_k(f8) * Cfg<false, 4, kNarrowN>::kSub;
    if (epi_warps == 8) return tcgen05_block_k(f8) * (pair ? Cfg<true, 8>::kSub : Cfg<false, 8>::kSub);
    return tcgen05_block_k(f8) * (pair ? Cfg<true, 4>::kSub : Cfg<false, 4>::kSub);
}
int tcgen05_load_rows_b(int pair, int tile_n) { return pair ? tile_n / 2 : tile_n; }
int tcgen05_load_rows_a() { return kBM; }
int tcgen05_smem_bytes(int pair, int epi_warps, int tile_n) {
    if (tile_n == kNarrowN) return Cfg<false, 4, kNarrowN>::kSmemBytes;
    if (tile_n == kFitN) return Cfg<true, 4, kFitN>::kSmemBytes;
    if (pair) return epi_warps == 8 ? Cfg<true, 8>::kSmemBytes : Cfg<true, 4>::kSmemBytes;
    return epi_warps == 8 ? Cfg<false, 8>::kSmemBytes : Cfg<false, 4>::kSmemBytes;
}
int tcgen05_stages(int pair, int epi_warps, int tile_n) {
    if (tile_n == kNarrowN) return Cfg<false, 4, kNarrowN>::kStages;
    if (tile_n == kFitN) return Cfg<true, 4, kFitN>::kStages;
    if (pair) return epi_warps == 8 ? Cfg<true, 8>::kStages : Cfg<true, 4>::kStages;
    return epi_warps == 8 ? Cfg<false, 8>::kStages : Cfg<false, 4>::kStages;
}

cudaError_t launch_k0(int out, void* D, const void* C, int M, int N, int64_t ldc, int64_t ldd, float alpha,
                      float beta, int has_c, int num_sms, cudaStream_t stream) {
    const int64_t total = (int64_t)M * N;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const dim3 grid((unsigned)blocks), block(256);
    if (out == kOutF32)
        return launch_with_pdl(gemm_k0_kernel<kOutF32>, grid, block, stream, D, C, M, N, ldc, ldd, alpha, beta, has_c);
    if (out == kOutF16)
        return launch_with_pdl(gemm_k0_kernel<kOutF16>, grid, block, stream, D, C, M, N, ldc, ldd, alpha, beta, has_c);
    return launch_with_pdl(gemm_k0_kernel<kOutBF16>, grid, block, stream, D, C, M, N, ldc, ldd, alpha, beta, has_c);
}

}  // namespace gb300
