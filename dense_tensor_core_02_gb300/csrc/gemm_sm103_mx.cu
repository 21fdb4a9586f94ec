// The MX block-scaled variant of the tcgen05 kernel (gemm_tcgen05.cuh with
// kMX: tcgen05.mma kind::mxf8f6f4, one UE8M0 scale per 32 K elements of each
// row of A and column of B, scales moved into tensor memory by tcgen05.cp),
// and the small kernel that puts the caller's scales into the order the
// main kernel loads them.  A translation unit of its own, so that it
// compiles in parallel with the others.
#include "gemm_tcgen05.cuh"

namespace gb300 {

cudaError_t prepare_kernels_mx() {
    cudaError_t e;
    if ((e = prepare_mx_group<false, false>()) != cudaSuccess) return e;
    if ((e = prepare_mx_group<false, true>()) != cudaSuccess) return e;
    if ((e = prepare_mx_group<true, false>()) != cudaSuccess) return e;
    return prepare_mx_group<true, true>();
}

cudaError_t launch_tcgen05_mx(const TcgenLaunch& L, cudaStream_t stream) {
    if (L.pair) return L.p.has_c ? launch_mx_group<true, true>(L, stream) : launch_mx_group<true, false>(L, stream);
    return L.p.has_c ? launch_mx_group<false, true>(L, stream) : launch_mx_group<false, false>(L, stream);
}

int tcgen05_mx_tile_n(int f32_out) { return f32_out ? kMxTileNF32 : kMxTileN; }
int tcgen05_mx_smem_bytes(int pair, int f32_out) {
    if (f32_out)
        return pair ? Cfg<true, 4, kMxTileNF32, true>::kSmemBytes : Cfg<false, 4, kMxTileNF32, true>::kSmemBytes;
    return pair ? Cfg<true, 4, kMxTileN, true>::kSmemBytes : Cfg<false, 4, kMxTileN, true>::kSmemBytes;
}
int tcgen05_mx_stages(int pair, int f32_out) {
    if (f32_out) return pair ? Cfg<true, 4, kMxTileNF32, true>::kStages : Cfg<false, 4, kMxTileNF32, true>::kStages;
    return pair ? Cfg<true, 4, kMxTileN, true>::kStages : Cfg<false, 4, kMxTileN, true>::kStages;
}

// One thread per (stage kc, tile, 128-row group g, row r of the group): the
// row's four scales of the stage (blocks 4 kc .. 4 kc + 3) become one 32-bit
// word at byte (r % 32) * 16 + (r / 32) * 4 of the group's 512-byte chunk,
// block 4 kc + j in byte j.  That is the layout tcgen05.cp .32x128b.warpx4
// reads: 32 rows of 16 bytes, row r % 32 holding rows r % 32 + 32 q of the
// group in its four words q.
__global__ void sf_tiles_kernel(uint32_t* out, const uint8_t* in, int64_t ld, int64_t rows, int64_t kblocks,
                                int tile_rows, int groups, int64_t tiles, int64_t total) {
    ptx::grid_dependency_wait();   // the previous kernel's writes are visible (programmatic launch)
    ptx::launch_dependents();
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(idx % 128);
        const int64_t chunk = idx / 128;   // ((kc * tiles + tile) * groups + g)
        const int g = (int)(chunk % groups);
        const int64_t tile = (chunk / groups) % tiles;
        const int64_t kc = chunk / groups / tiles;
        const int in_tile = g * 128 + r;
        const int64_t row = tile * tile_rows + in_tile;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t kb = kc * 4 + j;
            const uint32_t v = (in_tile < tile_rows && row < rows && kb < kblocks) ? in[row * ld + kb] : 127u;
            word |= v << (8 * j);
        }
        out[chunk * (kSfChunkBytes / 4) + (r % 32) * 4 + r / 32] = word;
    }
}

int64_t sf_tiles_bytes(int tile_rows, int64_t tiles, int64_t kchunks) {
    const int groups = (tile_rows + 127) / 128;
    return kchunks * tiles * groups * kSfChunkBytes;
}

cudaError_t launch_sf_tiles(uint8_t* out, const uint8_t* in, int64_t ld, int64_t rows, int64_t kblocks,
                            int tile_rows, int64_t tiles, int64_t kchunks, cudaStream_t stream) {
    const int groups = (tile_rows + 127) / 128;
    const int64_t total = kchunks * tiles * groups * 128;
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    return launch_with_pdl(sf_tiles_kernel, dim3((unsigned)blocks), dim3(256), stream,
                           reinterpret_cast<uint32_t*>(out), in, ld, rows, kblocks, tile_rows, groups, tiles, total);
}

}  // namespace gb300
