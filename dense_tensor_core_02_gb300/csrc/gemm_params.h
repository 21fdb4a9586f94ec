// Parameters shared by the host launcher and the sm_103a GEMM kernels, and
// the persistent tile scheduler (host-callable so it can be checked on CPU).
#pragma once
#include <cstdint>

#ifndef __CUDACC__
#define GB300_HD inline
#else
#define GB300_HD __host__ __device__ __forceinline__
#endif

namespace gb300 {

// Device-side status block: the first wait that gives up records itself here.
struct DeviceStatus {
    int code;     // 0 = ok, else a GEMM_ERR_* value
    int block;    // blockIdx.x of the reporting CTA
    int site;     // which wait gave up (WaitSite)
    int detail;   // tile index or chunk where it happened
};

enum WaitSite : int {
    kSiteProducerEmpty = 1,
    kSiteProducerTail = 2,
    kSiteMmaTmemEmpty = 3,
    kSiteMmaFull = 4,
    kSiteEpilogueTmemFull = 5,
    kSiteEpilogueC = 6,
};

struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, num_k_blocks, num_tiles;
    int32_t group_m;        // rasterisation: M tiles per group
    float alpha, beta;
    uint32_t idesc;         // tcgen05 instruction descriptor (kind::f16)
    int32_t a_mn_major;     // A stored [K, M] (transA): M contiguous
    int32_t b_mn_major;     // B stored [K, N] (no transB): N contiguous
    int32_t has_c;          // beta != 0: C is read
    int32_t skip_first_stage;  // test hook: never fill stage 0 of the first tile, so
                               // the MMA's wait on it runs out (bounded) and is reported
    uint64_t timeout_ns;    // bound on every in-kernel wait
    DeviceStatus* status;
    // A TMA store writes whole 16-byte pieces of a row even where they
    // straddle the tensor's last column, so D's tensor map covers only the
    // columns [0, n_tma) (n_tma = N rounded down to 16 bytes); the last
    // N - n_tma columns of each row are stored element by element.
    int32_t n_tma;
    int32_t pad0;
    void* d_ptr;
    int64_t ldd;            // D row stride in elements
    // L2 eviction priority of the TMA copies of A, B (loads) and D (stores):
    // 0 normal, 1 evict-first, 2 evict-last.
    int32_t hint_a, hint_b, hint_d;
    // Pause (ns) after each epilogue store chunk, except on a CTA's last
    // tile: spreads the D writes of all SMs over the next tile's main loop
    // instead of a simultaneous burst that stalls the operand loads.
    int32_t epi_pace_ns;
};

// Persistent-tile order with L2-friendly grouping: tiles run down a group of
// `group_m` M-tiles before moving to the next N column, so concurrently
// running tiles share A row panels and B column panels in L2.
GB300_HD void tile_coords(int tile, int num_m, int num_n, int group_m, int* m_blk, int* n_blk) {
    const int per_group = group_m * num_n;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int rows = (num_m - first_m) < group_m ? (num_m - first_m) : group_m;
    const int r = tile - g * per_group;
    *m_blk = first_m + r % rows;
    *n_blk = r / rows;
}

}  // namespace gb300
