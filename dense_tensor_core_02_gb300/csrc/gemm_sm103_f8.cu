// Instantiations of the tcgen05 kernel (gemm_tcgen05.cuh) for 8-bit
// floating-point operands, E4M3 / E5M2 (tcgen05.mma kind::f8f6f4), in a
// translation unit of their own so that they compile in parallel with the
// fp16 / bf16 ones.
#include "gemm_tcgen05.cuh"

namespace gb300 {

cudaError_t prepare_kernels_f8() { return prepare_family<true>(); }

cudaError_t launch_tcgen05_f8(const TcgenLaunch& L, cudaStream_t stream) { return launch_family<true>(L, stream); }

}  // namespace gb300
