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
    kSiteStreamK = 7,   // the stream-K arrival counter could not be updated
};

struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, num_k_blocks, num_tiles;
    int32_t group_m;        // rasterisation: M tiles per group
    float alpha, beta;
    uint32_t idesc;         // tcgen05 instruction descriptor (kind::f16, f8f6f4 or mxf8f6f4)
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
    int32_t pad0;           // keeps d_ptr 8-byte aligned
    void* d_ptr;
    int64_t ldd;            // D row stride in elements
    // L2 eviction priority of the TMA copies of A, B (loads) and D (stores):
    // 0 normal, 1 evict-first, 2 evict-last.
    int32_t hint_a, hint_b, hint_d;
    // Pause (ns) after each epilogue store chunk, except on a CTA's last
    // tile: spreads the D writes of all SMs over the next tile's main loop
    // instead of a simultaneous burst that stalls the operand loads.
    int32_t epi_pace_ns;
    // Stream-K (see Schedule): the trailing sk_tiles tiles are split along K.
    int32_t sk_tiles;
    int32_t ws_max_nc;        // partial slots per stream-K tile
    uint32_t ws_epoch;        // tags this launch's arrivals on the counters (24 bits used)
    int32_t pad2;           // keeps ws_counters 8-byte aligned
    uint32_t* ws_counters;    // [sk_tiles][2 CTA ranks] arrival counters
    void* ws_partials;        // [sk_tiles][ws_max_nc][2 ranks] x one CTA's fp32 accumulator (128 x tile N)
    // MX block scales (kernels with block scaling only), rearranged by the
    // host into 512-byte chunks, the rows of the SFA / SFB tensor maps.  A
    // chunk holds the scales of 128 rows (columns) for one 128-K sub-block:
    // byte (r % 32) * 16 + (r / 32) * 4 + j is row r's scale of block 4 kc
    // + j.  SFA chunk of 128-K sub-block kc and 128-row group g: row
    // kc * sf_a_groups + g.  SFB chunks of sub-block kc and N tile nb: the
    // (tile N / 128) rows from (kc * num_n_tiles + nb) * (tile N / 128) on.
    int32_t sf_a_groups;      // 128-row groups per sub-block in the SFA map (M tiles x CTAs per tile)
    // 1: packed E2M1 operands.  TMA's 16U4_ALIGN16B copies fill each 128-byte
    // shared row with 64 bytes of data (8 bytes per 16-byte group) and count
    // only those toward the barrier's transaction bytes.
    int32_t operands_packed4;
    // How the producer fetches one pipeline stage of A and of B: 2 = one 2-D
    // TMA box per 64-wide K sub-block (and per 64-wide MN chunk of an
    // MN-major operand); 3 = the whole stage of a K-major operand in one 3-D
    // box; 4 = the whole stage of an MN-major operand in one 4-D box.  Fewer
    // copies per stage measured 0.6 to 1 % faster on the tensor-bound shapes.
    // The whole-stage boxes serve stages [0, *_whole_stages) (their own
    // maps); later stages (a partial last one) take the 2-D boxes.
    int32_t a_box_dims, b_box_dims;
    int32_t a_whole_stages, b_whole_stages;
};

// ---------------------------------------------------------------------------
// Work schedule (host and device).  A tile's K loop has `iters` pipeline
// stages.  The first `num_tiles - sk_tiles` tiles (in raster order) are
// whole units, dealt round-robin to the `workers` persistent clusters; the
// last `sk_tiles` tiles ("stream-K" tiles) are cut along K so that every
// worker gets the same number of stages: worker w owns the positions
// [bound(w), bound(w+1)) of the sk_tiles * iters stream-K stages.  A tile
// cut between several workers is finished by whichever of them arrives last
// (it adds the others' partial accumulators), so no worker ever waits for
// another.

struct WorkUnit {
    int tile;   // tile index in raster order
    int kb;     // first pipeline stage of the unit
    int ke;     // one past its last stage
    int sk;     // index among the stream-K tiles, or -1 for a whole tile
    int ci;     // this worker's contributor index for the tile (0 = lowest K)
    int nc;     // number of contributors (1: no partials to combine)
};

struct Schedule {
    int num_tiles;
    int iters;      // pipeline stages per tile
    int workers;    // persistent clusters
    int sk_tiles;   // trailing tiles split along K (0: plain data-parallel)

    GB300_HD int dp_tiles() const { return num_tiles - sk_tiles; }
    GB300_HD int64_t sk_total() const { return (int64_t)sk_tiles * iters; }
    GB300_HD int64_t bound(int w) const { return sk_total() * w / workers; }
    // The worker whose stream-K range holds position pos (0 <= pos < sk_total).
    GB300_HD int worker_of(int64_t pos) const {
        int w = (int)(pos * workers / sk_total());
        while (w + 1 < workers && bound(w + 1) <= pos) ++w;
        while (w > 0 && bound(w) > pos) --w;
        return w;
    }
};

// Iterates the units of one worker: its stream-K segments first, then its
// whole tiles.
struct UnitIter {
    int64_t pos, end;   // remaining stream-K positions
    int dp_next;        // next whole tile

    GB300_HD void start(const Schedule& s, int w) {
        pos = s.sk_tiles ? s.bound(w) : 0;
        end = s.sk_tiles ? s.bound(w + 1) : 0;
        dp_next = w;
    }
    GB300_HD bool next(const Schedule& s, int w, WorkUnit* u) {
        if (pos < end) {
            const int t = (int)(pos / s.iters);
            const int64_t t0 = (int64_t)t * s.iters;
            const int64_t t1 = t0 + s.iters;
            const int64_t stop = end < t1 ? end : t1;
            const int first = s.worker_of(t0);
            const int last = s.worker_of(t1 - 1);
            u->tile = s.dp_tiles() + t;
            u->kb = (int)(pos - t0);
            u->ke = (int)(stop - t0);
            u->sk = t;
            u->ci = w - first;
            u->nc = last - first + 1;
            pos = stop;
            return true;
        }
        if (dp_next < s.dp_tiles()) {
            u->tile = dp_next;
            u->kb = 0;
            u->ke = s.iters;
            u->sk = -1;
            u->ci = 0;
            u->nc = 1;
            dp_next += s.workers;
            return true;
        }
        return false;
    }
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
