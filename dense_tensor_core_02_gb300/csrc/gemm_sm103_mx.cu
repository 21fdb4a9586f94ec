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

// The block scales in the order the main kernel loads them.  For each
// 128-K sub-block kc, tile and 128-row group g of the tile, a 512-byte chunk
// whose 32-bit word (r % 32) * 4 + r / 32 holds row r's four scales of the
// sub-block (blocks 4 kc .. 4 kc + 3, block 4 kc + j in byte j): the layout
// tcgen05.cp .32x128b.warpx4 reads, 32 rows of 16 bytes, row r % 32 holding
// rows r % 32 + 32 q of the group in its four words q.  Rows past the
// operand or the tile, and blocks past K, get 127 (a scale of 1).
//
// A thread block takes one group and a run of kSfRun sub-blocks: it gathers
// the run's scales row by row (each row's bytes are contiguous in the
// caller's array) into shared memory, then writes the run's chunks whole.
// Both operands' scales go in one launch: blocks [0, a.blocks) take SFA.
constexpr int kSfRun = 8;

__global__ void __launch_bounds__(256) sf_tiles_kernel(SfJob a, SfJob b) {
    ptx::grid_dependency_wait();   // the previous kernel's writes are visible (programmatic launch)
    ptx::launch_dependents();
    __shared__ uint32_t words[128 * (kSfRun + 1)];   // [row][sub-block of the run], one word of padding per row
    const int64_t bid = (int64_t)blockIdx.x;
    const bool is_a = bid < a.blocks;
    const SfJob& j = is_a ? a : b;
    const int64_t blk = is_a ? bid : bid - a.blocks;
    const int64_t runs = (j.kchunks + kSfRun - 1) / kSfRun;
    const int64_t run = blk % runs;
    const int g = (int)((blk / runs) % j.groups);
    const int64_t tile = blk / runs / j.groups;
    const int64_t kc0 = run * kSfRun;
    for (int i = threadIdx.x; i < 128 * kSfRun; i += blockDim.x) {
        const int r = i / kSfRun, c = i % kSfRun;
        const int in_tile = g * 128 + r;
        const int64_t row = tile * j.tile_rows + in_tile;
        const bool row_ok = in_tile < j.tile_rows && row < j.rows;
        uint32_t word = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t kb = (kc0 + c) * 4 + q;
            const uint32_t v = (row_ok && kb < j.kblocks) ? j.in[row * j.ld + kb] : 127u;
            word |= v << (8 * q);
        }
        words[r * (kSfRun + 1) + c] = word;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 128 * kSfRun; i += blockDim.x) {
        const int c = i / 128, p = i % 128;
        const int64_t kc = kc0 + c;
        if (kc >= j.kchunks) break;   // c only grows along a thread's loop
        const int r = (p & 3) * 32 + (p >> 2);
        j.out[((kc * j.tiles + tile) * j.groups + g) * 128 + p] = words[r * (kSfRun + 1) + c];
    }
}

int64_t sf_tiles_bytes(int tile_rows, int64_t tiles, int64_t kchunks) {
    const int groups = (tile_rows + 127) / 128;
    return kchunks * tiles * groups * kSfChunkBytes;
}

SfJob sf_job(uint8_t* out, const uint8_t* in, int64_t ld, int64_t rows, int64_t kblocks, int tile_rows, int64_t tiles,
             int64_t kchunks) {
    SfJob j{};
    j.out = reinterpret_cast<uint32_t*>(out);
    j.in = in;
    j.ld = ld;
    j.rows = rows;
    j.kblocks = kblocks;
    j.tile_rows = tile_rows;
    j.groups = (tile_rows + 127) / 128;
    j.tiles = tiles;
    j.kchunks = kchunks;
    j.blocks = kchunks > 0 ? tiles * j.groups * ((kchunks + kSfRun - 1) / kSfRun) : 0;
    return j;
}

cudaError_t launch_sf_tiles(const SfJob& a, const SfJob& b, cudaStream_t stream) {
    const int64_t blocks = a.blocks + b.blocks;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
    return launch_with_pdl(sf_tiles_kernel, dim3((unsigned)blocks), dim3(256), stream, a, b);
}

}  // namespace gb300
