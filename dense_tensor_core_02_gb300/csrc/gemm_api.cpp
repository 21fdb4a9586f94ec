// C-ABI entry points of libgemm_gb300.so (declared in include/gemm_gb300.h).
//
// Host side of the boundary: argument validation (every rejection happens
// before anything is enqueued), per-device state, TMA descriptor encoding,
// kernel selection and launch.  Nothing here synchronises the caller's
// stream except gemm_poll_device_error().
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/gemm_gb300.h"
#include "gemm_internal.h"
#include "gemm_params.h"

namespace {

using gb300::DeviceStatus;
using gb300::GemmParams;
using gb300::TcgenLaunch;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = 2147483647;           // TMA coordinates are signed 32-bit
constexpr int64_t kMaxStrideBytes = 1ll << 40;    // TMA global stride limit

struct DeviceState {
    bool ready = false;       // set-up done and succeeded
    int num_sms = 0;
    DeviceStatus* d_status = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

bool log_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("GEMM_LOG");
        return v && *v && std::strcmp(v, "0") != 0;
    }();
    return on;
}

#define GEMM_LOGF(...)                                \
    do {                                              \
        if (log_enabled()) {                          \
            std::fprintf(stderr, "[gemm_gb300] " __VA_ARGS__); \
            std::fputc('\n', stderr);                 \
        }                                             \
    } while (0)

int reject(int code, const char* why) {
    GEMM_LOGF("rejected (%s): %s", gemm_status_string(code), why);
    return code;
}

// Bound on every in-kernel wait (GEMM_WAIT_TIMEOUT_NS, default 2 s).
uint64_t wait_timeout_ns() {
    const char* v = std::getenv("GEMM_WAIT_TIMEOUT_NS");
    if (v && *v) {
        unsigned long long x = std::strtoull(v, nullptr, 10);
        if (x > 0) return (uint64_t)x;
    }
    return (uint64_t)2000000000ull;
}

// Test hook (GEMM_TEST_SKIP_FIRST_STAGE=1): the producer leaves stage 0 of
// the first tile empty, so the MMA's wait for it runs out after the time
// bound and the kernel reports GEMM_ERR_DEVICE_TIMEOUT without faulting.
int skip_first_stage_setting() {
    const char* v = std::getenv("GEMM_TEST_SKIP_FIRST_STAGE");
    return (v && std::strcmp(v, "1") == 0) ? 1 : 0;
}

// Test hook (GEMM_TEST_FAIL_SETUP=1): a device's one-time set-up fails
// before any CUDA call, as a transient failure would, so that tests can
// check that the failure is not cached and the next call sets up.
bool fail_setup_setting() {
    const char* v = std::getenv("GEMM_TEST_FAIL_SETUP");
    return v && std::strcmp(v, "1") == 0;
}

// Kernel variant: "pair" (256 x 256 tiles on 2 SMs), "single" (128 x 256),
// "narrow" (128 x 64) or automatic.
enum Variant { kAuto = -1, kSingle = 0, kPairV = 1, kNarrow = 2 };
int variant_override() {
    const char* v = std::getenv("GEMM_VARIANT");
    if (!v) return kAuto;
    if (std::strcmp(v, "pair") == 0) return kPairV;
    if (std::strcmp(v, "single") == 0) return kSingle;
    if (std::strcmp(v, "narrow") == 0) return kNarrow;
    return kAuto;
}

// Tile rasterisation: groups of this many tile rows, column by column
// (GEMM_GROUP_M overrides).  Deep tiles (more than 8 K-stages) re-read their
// operand panels from L2, and 8 rows per group keep a wave's panels resident
// (8192^3: 8 beats 4, 16 and 32; 8192^2 x 4096: 2 loses 7 %).  Shallow tiles
// are bound by their D stores, and 2 rows per group make a wave's stores
// cover whole rows of D (8192^2 x 1024: +3 %; x 256: +0.5 %).
int group_m_setting(int k_blocks) {
    const char* v = std::getenv("GEMM_GROUP_M");
    if (v && *v) {
        int g = std::atoi(v);
        if (g >= 1 && g <= 4096) return g;
    }
    return k_blocks <= 8 ? 2 : 8;
}

// SMs the persistent grid may use: all of the device's, or fewer when
// GEMM_MAX_SMS is set (at least 2), leaving the rest to other work on the
// GPU.
int plan_sms(int device_sms) {
    const char* v = std::getenv("GEMM_MAX_SMS");
    if (v && *v) {
        const int n = std::atoi(v);
        if (n >= 2 && n < device_sms) return n;
    }
    return device_sms;
}

// Memory-system tuning of a launch (needs the tile counts set).
//  * L2 eviction priorities of the A, B loads and D stores (0 normal, 1
//    evict-first, 2 evict-last).  Operand panels are re-read by the other
//    tiles of their row / column group, D is written once and never re-read:
//    A and B default to evict-last, D to evict-first.  A panel that only one
//    tile reads (A when there is a single tile column, B when there is a
//    single tile row) streams through once: evict-first (32768 x 256 x 4096:
//    +2.8 %).  GEMM_L2_HINTS="a,b,d" overrides.
//  * Epilogue pacing (GEMM_EPI_PACE_NS overrides): the persistent CTAs run
//    their tiles nearly in step, so without a pause every SM would store its
//    finished tile at the same moment, and the D stores would crowd out the
//    next tile's operand loads.  With two accumulators an epilogue has the
//    whole next main loop to finish in, so for tiles with a long main loop
//    (>= 24 stages, ~0.7 us each) each store chunk is followed by a pause of
//    20 ns per stage (a quarter of the main loop spread over a warp's 8
//    chunks), at most 2 us.  Measured (8192 x 8192, K = 4096 / 8192 / 16384):
//    +2 % / +1 % / +0.7 %; block-scaled 8192^3 (224-wide tiles): +2.7 % E4M3,
//    +2 % E2M1.  Tiles of 8 to 23 stages get 30 ns per stage (8192^2 x 1024,
//    8 stages: 240 ns, +1.5 %; 480 ns +0.9 %, 960 ns -29 %); shorter tiles
//    are store-bound and lose with any pause (K = 256: 150 ns -4 %).
void tuning(GemmParams& p, int tile_n) {
    p.hint_a = p.num_n_tiles == 1 ? 1 : 2;
    p.hint_b = p.num_m_tiles == 1 ? 1 : 2;
    p.hint_d = 1;
    const char* v = std::getenv("GEMM_L2_HINTS");
    int a, b, d;
    if (v && std::sscanf(v, "%d,%d,%d", &a, &b, &d) == 3 && a >= 0 && a <= 2 && b >= 0 && b <= 2 && d >= 0 &&
        d <= 2) {
        p.hint_a = a;
        p.hint_b = b;
        p.hint_d = d;
    }
    p.epi_pace_ns = 0;
    if (tile_n >= 192 && p.num_k_blocks >= 8)
        p.epi_pace_ns = std::min(2000, p.num_k_blocks * (p.num_k_blocks >= 24 ? 20 : 30));
    const char* pv = std::getenv("GEMM_EPI_PACE_NS");
    if (pv && *pv) {
        const int ns = std::atoi(pv);
        if (ns >= 0 && ns <= 100000) p.epi_pace_ns = ns;
    }
}

bool is_f8(int dtype) { return dtype == GEMM_E4M3 || dtype == GEMM_E5M2; }
// Bytes per element; packed E2M1 (two per byte) counts as 1 where a byte
// granularity is asked (alignment), and its rows are addressed through
// row_bytes().
int elem_size(int dtype) { return dtype == GEMM_F32 ? 4 : (is_f8(dtype) || dtype == GEMM_E2M1) ? 1 : 2; }
int64_t row_bytes(int dtype, int64_t elems) { return dtype == GEMM_E2M1 ? elems / 2 : elems * elem_size(dtype); }
int out_kind_of(int out_dtype) {
    return out_dtype == GEMM_F32 ? gb300::kOutF32 : out_dtype == GEMM_F16 ? gb300::kOutF16 : gb300::kOutBF16;
}

// Byte range [lo, hi) covered by a row-major rows x cols matrix.
void byte_range(const void* p, int64_t rows, int64_t cols, int64_t ld, int esz, uintptr_t* lo, uintptr_t* hi) {
    *lo = reinterpret_cast<uintptr_t>(p);
    *hi = *lo + (uintptr_t)(((rows - 1) * ld + cols) * esz);
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

// True while `s` is being captured into a CUDA graph: no allocation, no
// synchronising call may happen then.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

bool device_ready(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mutex);
    return g_devices[dev].ready;
}

// The one-time set-up of `dev` (the current device).  Only a successful
// set-up is kept: after a failure (reported to that call) the next call
// tries again.
int device_state(int dev, DeviceState** out) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0, status = GEMM_OK;
        DeviceStatus* d_status = nullptr;
        if (fail_setup_setting()) {
            status = GEMM_ERR_CUDA;
        } else if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            status = GEMM_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            GEMM_LOGF("device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
            status = GEMM_ERR_ARCH;
        } else if (gb300::prepare_kernels_on_current_device() != cudaSuccess) {
            status = GEMM_ERR_CUDA;
        } else if (cudaMalloc(&d_status, sizeof(DeviceStatus)) != cudaSuccess ||
                   cudaMemset(d_status, 0, sizeof(DeviceStatus)) != cudaSuccess) {
            status = GEMM_ERR_CUDA;
        }
        if (status != GEMM_OK) {
            if (d_status) cudaFree(d_status);
            cudaGetLastError();   // do not leave a sticky-free error behind
            return status;
        }
        st.num_sms = sms;
        st.d_status = d_status;
        st.ready = true;
    }
    *out = &st;
    return GEMM_OK;
}

// gemm()'s status record on `dev` if its set-up has run and succeeded,
// else NULL (nothing is created).
DeviceStatus* gemm_status_record(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    const DeviceState& st = g_devices[dev];
    return st.ready ? st.d_status : nullptr;
}

DeviceStatus* noalloc_status_record(int dev);   // gemm_noalloc()'s, defined with it below

int get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else
            cudaGetLastError();
    });
    return g_encode ? GEMM_OK : GEMM_ERR_CUDA;
}

// TMA moves bits: 8-bit floating-point operands travel as bytes.
CUtensorMapDataType tma_dtype(int dt) {
    switch (dt) {
        case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        case GEMM_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        // packed E2M1: each 16-element (8-byte) group lands in 16 bytes of
        // shared memory, the layout kind::mxf8f6f4 reads 4-bit operands in
        case GEMM_E2M1: return CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
        default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    }
}

// A 2-D row-major matrix: dim0 = contiguous extent, dim1 = rows; the box is
// box0 x box1 elements, staged with 128-byte swizzling, zero fill outside.
int encode_2d(CUtensorMap* map, int dt, const void* ptr, int64_t dim0, int64_t dim1, int64_t ld, uint32_t box0,
              uint32_t box1) {
    cuuint64_t dims[2] = {(cuuint64_t)dim0, (cuuint64_t)dim1};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes(dt, ld)};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, tma_dtype(dt), 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        GEMM_LOGF("cuTensorMapEncodeTiled failed (%d): dims %lld x %lld, ld %lld, box %u x %u", (int)r,
                  (long long)dim0, (long long)dim1, (long long)ld, box0, box1);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// One pipeline stage of a K-major operand (stored [rows][K], K contiguous)
// as a single box.  The K extent of each 128-byte shared row (bk elements)
// is the map's first dimension and the K chunks its third: dims {bk, rows,
// K / bk}, box {bk, box_rows, sub}; the box lands as `sub` consecutive
// {bk, box_rows} slabs, the image of `sub` 2-D boxes.  K is a multiple of
// bk (the caller's whole chunks).
int encode_kmajor_stage(CUtensorMap* map, int dt, const void* ptr, int64_t K, int64_t rows, int64_t ld, uint32_t bk,
                        uint32_t box_rows, uint32_t sub) {
    cuuint64_t dims[3] = {(cuuint64_t)bk, (cuuint64_t)rows, (cuuint64_t)(K / bk)};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes(dt, ld), (cuuint64_t)row_bytes(dt, bk)};
    cuuint32_t box[3] = {bk, box_rows, sub};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, tma_dtype(dt), 3, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        GEMM_LOGF("cuTensorMapEncodeTiled failed (%d): K-major stage map, K %lld, rows %lld, ld %lld", (int)r,
                  (long long)K, (long long)rows, (long long)ld);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// One pipeline stage of an MN-major operand (stored [K][mn], mn contiguous)
// as a single box: dims {64, bk, mn / 64, K / bk} (64 MN elements of a K
// row, the bk K rows of a sub-block, the 64-wide MN chunks, the sub-blocks),
// box {64, bk, box_mn / 64, sub}, landing as [sub-block][MN chunk][K row]:
// the image of the 2-D boxes {64, bk}.  mn and K are multiples of 64 and bk
// (the caller rounds mn up and K down; see describe_tcgen05).
int encode_mnmajor_stage(CUtensorMap* map, int dt, const void* ptr, int64_t mn, int64_t K, int64_t ld, uint32_t bk,
                         uint32_t box_mn, uint32_t sub) {
    cuuint64_t dims[4] = {64, (cuuint64_t)bk, (cuuint64_t)(mn / 64), (cuuint64_t)(K / bk)};
    cuuint64_t strides[3] = {(cuuint64_t)row_bytes(dt, ld), (cuuint64_t)row_bytes(dt, 64),
                             (cuuint64_t)row_bytes(dt, ld) * bk};
    cuuint32_t box[4] = {64, bk, box_mn / 64, sub};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, tma_dtype(dt), 4, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        GEMM_LOGF("cuTensorMapEncodeTiled failed (%d): MN-major stage map, mn %lld, K %lld, ld %lld", (int)r,
                  (long long)mn, (long long)K, (long long)ld);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// The rearranged MX scales (see GemmParams::sf_a_groups) as a 2-D tensor of
// 32-bit words: rows of 128 words (one 512-byte chunk), `box_rows` chunks
// per copy, no swizzle.
int encode_sf(CUtensorMap* map, const void* ptr, int64_t chunks, uint32_t box_rows) {
    cuuint64_t dims[2] = {128, (cuuint64_t)chunks};
    cuuint64_t strides[1] = {512};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        GEMM_LOGF("cuTensorMapEncodeTiled failed (%d) for the scales: %lld chunks, box %u", (int)r, (long long)chunks,
                  box_rows);
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

struct Plan {
    int pair;
    int tile_m, tile_n;
    int num_m, num_n, num_tiles;
    int grid;
    int smem;
    int epi_warps;
    int stages;
    int iters;         // pipeline stages per tile
    int sk_tiles;      // trailing tiles split along K (stream-K), 0 = data-parallel
    int max_nc;        // most contributors any stream-K tile has
    int64_t ws_bytes;  // workspace the stream-K fixup needs
};

// Wave-fitted 224-wide tiles (see make_plan): GEMM_FIT_TILES=0 never takes
// them, 1 takes them wherever they apply, unset chooses by wave count.
int fit_setting() {
    const char* v = std::getenv("GEMM_FIT_TILES");
    if (v && std::strcmp(v, "0") == 0) return 0;
    if (v && std::strcmp(v, "1") == 0) return 2;
    return 1;
}

// Stream-K policy: GEMM_STREAMK=0 never, 1 whenever the tiles do not fill
// whole waves; the default does the same.  A stream-K range shorter than
// GEMM_SK_MIN_ITERS stages (default 24) is not worth a partial: for small
// problems fewer clusters are used instead.
int streamk_setting() {
    const char* v = std::getenv("GEMM_STREAMK");
    return (v && std::strcmp(v, "0") == 0) ? 0 : 1;
}

// Measured on GB300: splitting pays only when each worker's stream-K share is
// long (8192^3: ~30 stages per worker, +1.3 %); short shares (4096^3: ~12)
// and memory-bound shapes lose more to the partial-tile traffic than they gain.
int sk_min_iters_setting() {
    const char* v = std::getenv("GEMM_SK_MIN_ITERS");
    if (v && *v) {
        const int n = std::atoi(v);
        if (n >= 1 && n <= 1 << 20) return n;
    }
    return 24;
}

constexpr int64_t kPartialBytes = 128 * 256 * 4;   // one CTA's 128 x 256 fp32 accumulator

// TMA (the tcgen05 kernel) needs 16-byte-aligned bases and row strides.
bool tma_layout_ok(const void* D, const void* A, const void* B, const void* C, int64_t K, int64_t lda, int64_t ldb,
                   int64_t ldc, int64_t ldd, int isz, int osz, bool has_c) {
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    bool ok = a16(D) && ((ldd * osz) & 15) == 0;
    if (has_c) ok = ok && a16(C) && ((ldc * osz) & 15) == 0;
    if (K > 0) ok = ok && a16(A) && a16(B) && (((lda * isz) | (ldb * isz)) & 15) == 0;
    return ok;
}

// The tcgen05 kernel stages 8-bit operands K-major only: A stored [M, K]
// (transA = 0) and B stored [N, K] (transB = 1).
bool operand_majors_ok(int in_dtype, int transA, int transB) { return !is_f8(in_dtype) || (!transA && transB); }

int64_t env_int64(const char* name, int64_t dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::strtoll(v, nullptr, 10) : dflt;
}

// Aligned fp16 / bf16 problems with a short K and a small D run soonest on
// the mma.sync route's atom kernel.  Graph-replayed device time per launch
// on GB300 (atom kernel vs tcgen05 kernel, us): 16x8x16 1.9 vs 2.8, 64x64x8
// 1.8 vs 3.1, 256x256x32 2.9 vs 3.1, 512x512x16 2.4 vs 3.2; from K = 64 on
// the tcgen05 kernel is as fast or faster (64^3 3.6 vs 3.0, 8x8x512 14.1 vs
// 4.6, 2048^2 x 8 14.4 vs 6.7).  GEMM_SYNC_MAX_WORK replaces the rule by
// M*N*K <= its value.
bool sync_pays(int64_t M, int64_t N, int64_t K) {
    const int64_t bound = env_int64("GEMM_SYNC_MAX_WORK", -1);
    if (bound >= 0) return M * N * K <= bound;
    return K <= 32 && M * N <= (int64_t)1 << 18;
}

// Which kernel:
//  * the tcgen05 kernel on the caller's buffers when it can take them as
//    they are (TMA's alignment rule; 8-bit operands K-major), except for
//    fp16 / bf16 problems so small that the mma.sync route's atom kernel
//    finishes sooner (sync_pays);
//  * otherwise, when the caller may allocate and the problem pays for the
//    copies (M*N*K > GEMM_REPACK_MIN_WORK, default 2^22; always for 8-bit
//    operands), the tcgen05 kernel on repacked copies (gemm_repacked);
//  * else the warp-level mma.sync kernel, which takes any element-aligned
//    fp16 / bf16 layout as it is; 8-bit operands have no such kernel.
// GEMM_PATH=tcgen05|mma_sync forces a kernel where one can run (tcgen05
// through the repacking when it cannot take the buffers as they are).
enum Route { kRouteTcgen05, kRouteRepack, kRouteSync, kRouteNone };
Route route_for(bool direct_ok, bool f8, bool can_allocate, int64_t M, int64_t N, int64_t K) {
    const char* v = std::getenv("GEMM_PATH");
    const int64_t work = M * N * K;
    if (!f8 && v && std::strcmp(v, "mma_sync") == 0) return kRouteSync;
    const bool force_tc = v && std::strcmp(v, "tcgen05") == 0;
    if (direct_ok) return (!f8 && !force_tc && sync_pays(M, N, K)) ? kRouteSync : kRouteTcgen05;
    if (can_allocate && (f8 || force_tc || work > env_int64("GEMM_REPACK_MIN_WORK", 1 << 22))) return kRouteRepack;
    return f8 ? kRouteNone : kRouteSync;
}

// Which kernel of the mma.sync route.  Graph-replayed device time per launch
// on GB300 (us; the one-warp-per-16x8-block atom kernel vs the tiled one):
// 16x8x16 1.6 vs 4.0, 128^3 5.9 vs 12.1, 256^3 10.9 vs 20.2, 1000x64x64 3.8 vs
// 6.8; the tiled kernel's shared-memory reuse wins once D is large
// (2048^2 x 8: 40.5 vs 11.1; 512^3: 42.8 vs 36.7).  GEMM_SYNC_ATOM_MAX_WORK
// replaces the rule by M*N*K <= its value.
bool sync_atom_kernel(int64_t M, int64_t N, int64_t K) {
    const int64_t bound = env_int64("GEMM_SYNC_ATOM_MAX_WORK", -1);
    if (bound >= 0) return M * N * K <= bound;
    return M * N <= (int64_t)1 << 18 && M * N * K <= (int64_t)1 << 24;
}

cudaError_t launch_sync(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float alpha,
                        float beta, int in_dtype, int out_kind, bool has_c, cudaStream_t s) {
    gb300::SyncParams sp;
    sp.A = A;
    sp.B = B;
    sp.C = has_c ? C : nullptr;
    sp.D = D;
    sp.M = M;
    sp.N = N;
    sp.K = K;
    sp.lda = lda;
    sp.ldb = ldb;
    sp.ldc = has_c ? ldc : 0;
    sp.ldd = ldd;
    sp.transA = transA;
    sp.transB = transB;
    sp.alpha = alpha;
    sp.beta = beta;
    sp.in_bf16 = in_dtype == GEMM_BF16 ? 1 : 0;
    sp.out = out_kind;
    sp.has_c = has_c ? 1 : 0;
    sp.atom = sync_atom_kernel(M, N, K) ? 1 : 0;
    return gb300::launch_mma_sync(sp, s);
}

// Epilogue warps: 8 when a tile's main loop is short (few K stages), so the
// time goes into storing D; 4 otherwise.  The 8-warp kernels exist for f32
// output only.  GEMM_EPI_WARPS=4|8 overrides (f32 output).
int epi_warps_for(int64_t K, int pair, int out_dtype, int tile_n, int f8) {
    if (out_dtype != GEMM_F32 || tile_n == gb300::tcgen05_narrow_n()) return 4;
    const char* v = std::getenv("GEMM_EPI_WARPS");
    if (v && (std::strcmp(v, "4") == 0 || std::strcmp(v, "8") == 0)) return std::atoi(v);
    const int64_t stage_k = gb300::tcgen05_stage_k(pair, f8, 4, tile_n);
    return (K + stage_k - 1) / stage_k <= 4 ? 8 : 4;
}

// mx: the block-scaled kernel, whose tiles are 224 wide for f32 D and 192
// for 16-bit D (on a CTA pair or one SM; no narrow tiles), with 4 epilogue
// warps; stream-K applies to it as to the others.  b_kmajor: B is stored
// [N, K] (transB), which the 224-wide wave-fitted tiles need.
Plan make_plan(int64_t M, int64_t N, int64_t K, int num_sms, bool allow_streamk, int out_dtype, int f8, int mx = 0,
               int b_kmajor = 0) {
    Plan pl{};
    const int ov = (mx && variant_override() == kNarrow) ? kAuto : variant_override();
    pl.pair = ov == kPairV || (ov == kAuto && M > gb300::tcgen05_tile_m(0)) ? 1 : 0;
    pl.tile_m = gb300::tcgen05_tile_m(pl.pair);
    pl.tile_n = mx ? gb300::tcgen05_mx_tile_n(out_dtype == GEMM_F32) : gb300::tcgen05_wide_n();
    // Narrow 128 x 64 tiles when the wide ones would keep at most a quarter
    // of the SMs busy (the time then goes into latency and into each CTA's
    // epilogue, which a narrow tile cuts by four), or when N fits one.
    const int64_t wide_ctas = ((M + pl.tile_m - 1) / pl.tile_m) * ((N + pl.tile_n - 1) / pl.tile_n) * (pl.pair + 1);
    if (!mx && (ov == kNarrow || (ov == kAuto && (wide_ctas * 4 <= num_sms || N <= gb300::tcgen05_narrow_n())))) {
        pl.pair = 0;
        pl.tile_m = gb300::tcgen05_tile_m(0);
        pl.tile_n = gb300::tcgen05_narrow_n();
    }
    pl.num_m = (int)((M + pl.tile_m - 1) / pl.tile_m);
    pl.num_n = (int)((N + pl.tile_n - 1) / pl.tile_n);
    pl.num_tiles = pl.num_m * pl.num_n;
    pl.epi_warps = mx ? 4 : epi_warps_for(K, pl.pair, out_dtype, pl.tile_n, f8);
    const int64_t stage_k = gb300::tcgen05_stage_k(pl.pair, f8, pl.epi_warps, pl.tile_n);
    pl.iters = (int)((K + stage_k - 1) / stage_k);
    const int units = pl.pair ? num_sms / 2 : num_sms;   // clusters that fit at once
    // Wave-fitted tiles: a persistent launch takes about (waves) x (time of
    // one tile), which grows with the tile width.  When the 256-wide tiles
    // leave the last wave partly empty and stream-K would not split it,
    // 224-wide ones can take fewer tile-widths in all (4096^2: 4 waves of
    // 256 columns, or 4 waves of 224).  CTA pairs with f32 D, K-major B and
    // the 4-warp epilogue; taken when that saves at least 5 %.
    const int fit = fit_setting();
    if (!mx && fit && pl.pair && b_kmajor && out_dtype == GEMM_F32 && pl.epi_warps == 4 &&
        pl.tile_n == gb300::tcgen05_wide_n()) {
        const int fit_n = gb300::tcgen05_fit_n();
        const int64_t n_fit = (N + fit_n - 1) / fit_n;
        const int64_t tiles_fit = (int64_t)pl.num_m * n_fit;
        const int64_t rem = pl.num_tiles % units;
        const bool sk_fills = allow_streamk && streamk_setting() && pl.iters > 0 && rem != 0 &&
                              pl.num_tiles > units && rem * pl.iters / units >= sk_min_iters_setting();
        const double waves_wide =
            sk_fills ? (double)pl.num_tiles / units : (double)((pl.num_tiles + units - 1) / units);
        const double cost_wide = waves_wide * gb300::tcgen05_wide_n();
        const double cost_fit = (double)((tiles_fit + units - 1) / units) * fit_n;
        if (fit == 2 || cost_fit < 0.95 * cost_wide) {
            pl.tile_n = fit_n;
            pl.num_n = (int)n_fit;
            pl.num_tiles = (int)tiles_fit;
        }
    }
    int clusters = pl.num_tiles < units ? pl.num_tiles : units;
    if (clusters < 1) clusters = 1;
    // Stream-K when the whole tiles leave the last wave partly empty.
    if (allow_streamk && streamk_setting() && pl.iters > 0 && pl.num_tiles % units != 0) {
        const int min_iters = sk_min_iters_setting();
        if (pl.num_tiles > units) {
            const int rem = pl.num_tiles % units;
            if ((int64_t)rem * pl.iters / units >= min_iters) {
                clusters = units;
                pl.sk_tiles = rem;
            }
        } else {
            const int64_t total = (int64_t)pl.num_tiles * pl.iters;
            const int64_t workers = std::min<int64_t>(units, total / min_iters);
            if (workers > pl.num_tiles) {
                clusters = (int)workers;
                pl.sk_tiles = pl.num_tiles;
            }
        }
    }
    pl.grid = pl.pair ? 2 * clusters : clusters;
    if (pl.sk_tiles > 0) {
        const gb300::Schedule s{pl.num_tiles, pl.iters, clusters, pl.sk_tiles};
        for (int t = 0; t < pl.sk_tiles; ++t) {
            const int nc = s.worker_of((int64_t)(t + 1) * pl.iters - 1) - s.worker_of((int64_t)t * pl.iters) + 1;
            pl.max_nc = std::max(pl.max_nc, nc);
        }
        const int64_t counters = ((int64_t)pl.sk_tiles * 2 * 4 + 255) / 256 * 256;
        pl.ws_bytes = counters + (int64_t)pl.sk_tiles * pl.max_nc * 2 * kPartialBytes;
    }
    if (mx) {
        pl.smem = gb300::tcgen05_mx_smem_bytes(pl.pair, out_dtype == GEMM_F32);
        pl.stages = gb300::tcgen05_mx_stages(pl.pair, out_dtype == GEMM_F32);
        return pl;
    }
    pl.smem = gb300::tcgen05_smem_bytes(pl.pair, pl.epi_warps, pl.tile_n);
    pl.stages = gb300::tcgen05_stages(pl.pair, pl.epi_warps, pl.tile_n);
    return pl;
}

// Device workspaces, one per (kind, device, stream): calls on one stream run
// in order, so they can share one; calls on different streams get different
// ones.  Grown on demand (freeing the old one synchronises the device) and
// kept until the process exits.  `epoch` numbers the launches that use it.
// Kinds: the stream-K partial sums and arrival counters, the repacked
// operands / outputs of gemm_repacked, gemm_mx's rearranged scales, and its
// copies of 4-bit operands padded to TMA's 4-bit rules.
enum WorkspaceKind { kWsStreamK = 0, kWsRepack = 1, kWsScales = 2, kWsFp4 = 3 };
struct Workspace {
    int kind;
    int dev;
    cudaStream_t stream;
    void* base;
    int64_t bytes;
    uint32_t epoch;
    bool captured;   // a CUDA graph captured a launch that uses `base`
};
std::vector<Workspace> g_workspaces;
// Buffers replaced while a captured graph may still use them: kept (not
// freed) until the process exits, so that replaying that graph stays safe.
std::vector<void*> g_retired;

// `may_grow` false (the stream is being captured into a CUDA graph, where
// allocating is not allowed): only an existing workspace that is large
// enough is returned; otherwise GEMM_ERR_CUDA, with nothing changed.  A
// workspace a capture has used is never freed when it grows later (graph
// replays keep using its address); others are freed (which synchronises
// the device, so no launch still uses them).
int workspace_for(int kind, int dev, cudaStream_t s, int64_t bytes, void** base, uint32_t* epoch, bool may_grow) {
    std::lock_guard<std::mutex> lock(g_mutex);
    Workspace* w = nullptr;
    for (auto& x : g_workspaces)
        if (x.kind == kind && x.dev == dev && x.stream == s) w = &x;
    if (!w) {
        g_workspaces.push_back(Workspace{kind, dev, s, nullptr, 0, 0, false});
        w = &g_workspaces.back();
    }
    if (w->bytes < bytes) {
        if (!may_grow) return GEMM_ERR_CUDA;
        if (w->base && w->captured) {
            g_retired.push_back(w->base);
        } else if (w->base && cudaFree(w->base) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        w->base = nullptr;
        w->bytes = 0;
        w->captured = false;
        if (cudaMalloc(&w->base, (size_t)bytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        w->bytes = bytes;
    }
    if (!may_grow) w->captured = true;
    w->epoch = (w->epoch + 1) & 0xFFFFFFu;
    *base = w->base;
    *epoch = w->epoch;
    return GEMM_OK;
}

// The argument rules shared by gemm() and gemm_noalloc(), checked on the
// host without touching the device.
int validate(const void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
             int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float beta, int in_dtype,
             int out_dtype) {
    if (in_dtype != GEMM_F16 && in_dtype != GEMM_BF16 && !is_f8(in_dtype))
        return reject(GEMM_ERR_UNSUPPORTED_DTYPE, "in_dtype");
    if (out_dtype != GEMM_F32 && out_dtype != GEMM_F16 && out_dtype != GEMM_BF16)
        return reject(GEMM_ERR_UNSUPPORTED_DTYPE, "out_dtype");
    if (M < 0 || N < 0 || K < 0) return reject(GEMM_ERR_INVALID_ARG, "negative size");
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return reject(GEMM_ERR_INVALID_ARG, "transpose flag not 0/1");
    if (M == 0 || N == 0) return GEMM_OK;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return reject(GEMM_ERR_TOO_LARGE, "dimension");
    const bool has_c = beta != 0.0f;
    const int isz = elem_size(in_dtype);
    const int osz = elem_size(out_dtype);
    if (!D) return reject(GEMM_ERR_INVALID_ARG, "D is NULL");
    if (ldd < N) return reject(GEMM_ERR_INVALID_ARG, "ldd < N");
    if (has_c) {
        if (!C) return reject(GEMM_ERR_INVALID_ARG, "C is NULL with beta != 0");
        if (ldc < N) return reject(GEMM_ERR_INVALID_ARG, "ldc < N");
    }
    if (K > 0) {
        if (!A || !B) return reject(GEMM_ERR_INVALID_ARG, "A or B is NULL");
        if (lda < (transA ? M : K)) return reject(GEMM_ERR_INVALID_ARG, "lda too small");
        if (ldb < (transB ? K : N)) return reject(GEMM_ERR_INVALID_ARG, "ldb too small");
        if (lda * isz >= kMaxStrideBytes || ldb * isz >= kMaxStrideBytes) return reject(GEMM_ERR_TOO_LARGE, "stride");
        if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & (uintptr_t)(isz - 1))
            return reject(GEMM_ERR_MISALIGNED, "A or B not element-aligned");
    }
    if (ldd * osz >= kMaxStrideBytes || (has_c && ldc * osz >= kMaxStrideBytes))
        return reject(GEMM_ERR_TOO_LARGE, "stride");
    if (reinterpret_cast<uintptr_t>(D) & (uintptr_t)(osz - 1)) return reject(GEMM_ERR_MISALIGNED, "D not element-aligned");
    if (has_c && (reinterpret_cast<uintptr_t>(C) & (uintptr_t)(osz - 1)))
        return reject(GEMM_ERR_MISALIGNED, "C not element-aligned");
    uintptr_t d0, d1;
    byte_range(D, M, N, ldd, osz, &d0, &d1);
    if (K > 0) {
        uintptr_t a0, a1, b0, b1;
        byte_range(A, transA ? K : M, transA ? M : K, lda, isz, &a0, &a1);
        byte_range(B, transB ? N : K, transB ? K : N, ldb, isz, &b0, &b1);
        if (overlaps(d0, d1, a0, a1) || overlaps(d0, d1, b0, b1)) return reject(GEMM_ERR_ALIAS, "D overlaps A or B");
    }
    if (has_c && !(C == D && ldc == ldd)) {
        uintptr_t c0, c1;
        byte_range(C, M, N, ldc, osz, &c0, &c1);
        if (overlaps(d0, d1, c0, c1)) return reject(GEMM_ERR_ALIAS, "D overlaps C (other than C == D, ldc == ldd)");
    }
    return GEMM_OK;
}

// gemm_mx's extra arguments: 8-bit operands; for K > 0 both scale arrays,
// rows of at least ceil(K/32) scales, neither overlapping D.  Called after
// validate() with M, N > 0.
int validate_scales(const void* D, const void* SFA, const void* SFB, int64_t M, int64_t N, int64_t K,
                    int64_t ld_sfa, int64_t ld_sfb, int64_t ldd, int out_dtype) {
    if (K == 0) return GEMM_OK;
    const int64_t kblocks = (K + 31) / 32;
    if (!SFA || !SFB) return reject(GEMM_ERR_INVALID_ARG, "SFA or SFB is NULL");
    if (ld_sfa < kblocks || ld_sfb < kblocks) return reject(GEMM_ERR_INVALID_ARG, "scale row shorter than ceil(K/32)");
    uintptr_t d0, d1, a0, a1, b0, b1;
    byte_range(D, M, N, ldd, elem_size(out_dtype), &d0, &d1);
    byte_range(SFA, M, kblocks, ld_sfa, 1, &a0, &a1);
    byte_range(SFB, N, kblocks, ld_sfb, 1, &b0, &b1);
    if (overlaps(d0, d1, a0, a1) || overlaps(d0, d1, b0, b1)) return reject(GEMM_ERR_ALIAS, "D overlaps SFA or SFB");
    return GEMM_OK;
}

// Tensor maps, kernel parameters and instruction descriptor of one tcgen05
// launch over buffers it can take as they are; the caller adds the status
// record and, for stream-K, the workspace.
int describe_tcgen05(TcgenLaunch* L, const Plan& pl, void* D, const void* A, const void* B, const void* C,
                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA,
                     int transB, float alpha, float beta, int in_dtype, int out_dtype) {
    const bool has_c = beta != 0.0f;
    const bool f8 = is_f8(in_dtype) || in_dtype == GEMM_E2M1;   // 128 K elements per 128-byte shared row
    const int osz = elem_size(out_dtype);
    int rc;
    if ((rc = get_encoder()) != GEMM_OK) return rc;
    std::memset(L, 0, sizeof(*L));
    // 224-wide tiles (wave-fitted or block-scaled) stage B K-major only
    if (pl.tile_n == gb300::tcgen05_fit_n() && !transB) return GEMM_ERR_INVALID_ARG;
    const uint32_t bk = (uint32_t)gb300::tcgen05_block_k(f8);   // K elements per 128-byte row
    // K sub-blocks per pipeline stage, and the rows of A and B one CTA stages
    const uint32_t sub = (uint32_t)(gb300::tcgen05_stage_k(pl.pair, f8, pl.epi_warps, pl.tile_n) / (int)bk);
    const uint32_t rows_a = (uint32_t)gb300::tcgen05_load_rows_a();
    const uint32_t rows_b = (uint32_t)gb300::tcgen05_load_rows_b(pl.pair, pl.tile_n);
    // A whole stage in one box for the kernels whose stages hold two K
    // sub-blocks (GEMM_STAGE_BOXES=0: always the 2-D boxes).  Measured
    // against the 2-D boxes: 8192^3 +0.6 to +0.8 %, 4096^3 bf16 beta = 1
    // +1.0 %, 8192^2 x 4096 +0.9 %, 512^3 -11 % time, 1000^3 -4 % time.
    // (The operand supply itself is not the limit: in this kernel's access
    // pattern TMA delivers ~95 bytes per SM clock on every SM with either
    // form, against the 64 the tensor pipe needs.)  The 8-epilogue-warp
    // kernel (one sub-block per stage, bound by its D stores) lost 1.7 % with
    // the MN-major chunks merged, and keeps them apart.
    //
    // The whole-stage maps cover only complete stages.  A K-major map counts
    // whole 128-byte K chunks, and a partial last stage takes the 2-D boxes:
    // a partial chunk would read on into the next row instead of reading
    // zeros.  An MN-major map counts 64-wide MN chunks; when M (or N) is not
    // a multiple of 64 the last chunk reads up to 63 elements past the end of
    // each K row, into the row after it.  Those elements only reach rows (or
    // columns) of D that are never stored, and the last K row, which has no
    // row after it, always comes through the 2-D boxes.  That takes an
    // extent of at least 64, so that the overrun stays inside the next row.
    const char* sb = std::getenv("GEMM_STAGE_BOXES");
    const bool boxes_ok = sub > 1 && !(sb && std::strcmp(sb, "0") == 0);
    const int64_t stage_k = (int64_t)bk * sub;
    const int64_t full_stages = K / stage_k;               // stages with every K chunk complete
    const int64_t all_stages = (K + stage_k - 1) / stage_k;
    // whole-stage count of an MN-major operand of extent mn (0: 2-D boxes only)
    auto mn_whole = [&](int64_t mn) -> int64_t {
        if (mn % 64 == 0) return full_stages;
        return mn >= 64 ? std::min(full_stages, all_stages - 1) : 0;
    };
    int a_dims = 2, b_dims = 2;
    int64_t a_whole = 0, b_whole = 0;
    // A: K-major (transA = 0) as [M rows][K], else MN-major as [K rows][M]
    if (!transA)
        rc = encode_2d(&L->a, in_dtype, A, K, M, lda, bk, rows_a);
    else
        rc = encode_2d(&L->a, in_dtype, A, M, K, lda, 64, bk);
    if (rc != GEMM_OK) return rc;
    if (boxes_ok && !transA && full_stages > 0) {
        a_dims = 3;
        a_whole = full_stages;
        rc = encode_kmajor_stage(&L->a_stage, in_dtype, A, K / bk * bk, M, lda, bk, rows_a, sub);
    } else if (boxes_ok && transA && mn_whole(M) > 0) {
        a_dims = 4;
        a_whole = mn_whole(M);
        rc = encode_mnmajor_stage(&L->a_stage, in_dtype, A, (M + 63) / 64 * 64, K / bk * bk, lda, bk, rows_a, sub);
    }
    if (rc != GEMM_OK) return rc;
    // B: K-major (transB = 1) as [N rows][K], else MN-major as [K rows][N]
    if (transB)
        rc = encode_2d(&L->b, in_dtype, B, K, N, ldb, bk, rows_b);
    else
        rc = encode_2d(&L->b, in_dtype, B, N, K, ldb, 64, bk);
    if (rc != GEMM_OK) return rc;
    if (boxes_ok && transB && full_stages > 0) {
        b_dims = 3;
        b_whole = full_stages;
        rc = encode_kmajor_stage(&L->b_stage, in_dtype, B, K / bk * bk, N, ldb, bk, rows_b, sub);
    } else if (boxes_ok && !transB && mn_whole(N) > 0) {
        b_dims = 4;
        b_whole = mn_whole(N);
        rc = encode_mnmajor_stage(&L->b_stage, in_dtype, B, (N + 63) / 64 * 64, K / bk * bk, ldb, bk, rows_b, sub);
    }
    if (rc != GEMM_OK) return rc;
    const uint32_t chunk_cols = 128u / (uint32_t)osz;
    // TMA stores write whole 16-byte pieces of a row, even past the tensor's
    // last column: D's map stops at the last whole piece (n_tma) and the
    // kernel stores columns [n_tma, N) element by element.
    const int64_t vec = 16 / osz;
    const int64_t n_tma = (N / vec) * vec;
    if ((rc = encode_2d(&L->d, out_dtype, D, n_tma > 0 ? n_tma : N, M, ldd, chunk_cols, 32)) != GEMM_OK) return rc;
    if (has_c && (rc = encode_2d(&L->c, out_dtype, C, N, M, ldc, chunk_cols, 32)) != GEMM_OK) return rc;
    GemmParams& p = L->p;
    p.M = (int32_t)M;
    p.N = (int32_t)N;
    p.K = (int32_t)K;
    p.a_box_dims = a_dims;
    p.b_box_dims = b_dims;
    p.a_whole_stages = (int32_t)a_whole;
    p.b_whole_stages = (int32_t)b_whole;
    p.num_m_tiles = pl.num_m;
    p.num_n_tiles = pl.num_n;
    p.num_k_blocks = (int32_t)all_stages;   // pipeline stages per tile
    p.num_tiles = pl.num_tiles;
    p.group_m = group_m_setting(p.num_k_blocks);
    p.alpha = alpha;
    p.beta = beta;
    p.a_mn_major = transA ? 1 : 0;
    p.b_mn_major = transB ? 0 : 1;
    p.has_c = has_c ? 1 : 0;
    p.timeout_ns = wait_timeout_ns();
    p.n_tma = (int32_t)n_tma;
    p.d_ptr = D;
    p.ldd = ldd;
    tuning(p, pl.tile_n);
    // tcgen05 instruction descriptor (kind::f16 or kind::f8f6f4, chosen by the
    // kernel instantiation): D format f32 (bits 4-5 = 1); A / B format (bits
    // 7-9, 10-12): kind::f16 0 = f16, 1 = bf16; kind::f8f6f4 0 = E4M3, 1 = E5M2;
    // A / B major (bits 15, 16: 1 = MN-major); N >> 3 (bits 17-22); M >> 4
    // (bits 24-28).
    const uint32_t fmt = (in_dtype == GEMM_BF16 || in_dtype == GEMM_E5M2) ? 1u : 0u;
    const uint32_t mma_m = (uint32_t)pl.tile_m;   // 128 (one SM) or 256 (CTA pair)
    p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)p.a_mn_major << 15) |
              ((uint32_t)p.b_mn_major << 16) | (((uint32_t)pl.tile_n >> 3) << 17) | ((mma_m >> 4) << 24);
    L->pair = pl.pair;
    L->tile_n = pl.tile_n;
    L->f8 = f8 ? 1 : 0;
    L->out = out_kind_of(out_dtype);
    L->grid = pl.grid;
    L->epi_warps = pl.epi_warps;
    // Programmatic dependent launch: the kernel's set-up overlaps the tail of
    // the previous kernel on the stream (GEMM_PDL=0 turns it off).
    L->pdl = gb300::pdl_setting();
    return GEMM_OK;
}

int launch_described(const TcgenLaunch& L, cudaStream_t s) {
    cudaError_t e = gb300::launch_tcgen05(L, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_LAUNCH, cudaGetErrorString(e));
    }
    return GEMM_OK;
}

int launch_k0_or_reject(int out_dtype, void* D, const void* C, int64_t M, int64_t N, int64_t ldc, int64_t ldd,
                        float alpha, float beta, int num_sms, cudaStream_t s) {
    const bool has_c = beta != 0.0f;
    cudaError_t e = gb300::launch_k0(out_kind_of(out_dtype), D, has_c ? C : nullptr, (int)M, (int)N, ldc, ldd, alpha,
                                     beta, has_c ? 1 : 0, num_sms, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_LAUNCH, cudaGetErrorString(e));
    }
    return GEMM_OK;
}

int launch_sync_or_reject(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float alpha,
                          float beta, int in_dtype, int out_dtype, cudaStream_t s) {
    cudaError_t e = launch_sync(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta, in_dtype,
                                out_kind_of(out_dtype), beta != 0.0f, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_LAUNCH, cudaGetErrorString(e));
    }
    return GEMM_OK;
}

// Layouts the tcgen05 kernel cannot take as they are, made so.  Each operand
// or output whose address or row stride is off the 16-byte grid is copied
// to (for D: computed in) workspace rows padded to 16 bytes; an 8-bit operand
// stored MN-major (A with transA, B without transB) is transposed into a
// K-major workspace copy.  The call then runs on the prepared buffers, and a
// workspace D is copied back.
//  * D misaligned: the kernel writes a workspace D'.  C, when read, is read
//    where it is if it is aligned and is not D; otherwise it is copied into
//    D' first and the kernel runs in place on D'.
//  * D aligned, C misaligned: C is copied into D, and the kernel runs in place.
// Returns kNoWorkspace (before enqueuing anything) when the workspace cannot
// be had, else GEMM_OK or the inner call's error.
constexpr int kNoWorkspace = 1;
// With SFA / SFB (block-scaled operands) the inner call is gemm_mx(); the
// scales are indexed by row of op(A) and column of op(B), so they need no
// repacking here.
int gemm_repacked(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float alpha,
                  float beta, int in_dtype, int out_dtype, int dev, cudaStream_t s, bool may_grow,
                  const void* SFA = nullptr, const void* SFB = nullptr, int64_t ld_sfa = 0, int64_t ld_sfb = 0) {
    // Packed 4-bit operands (K-major, K and the leading dimensions even) are
    // moved as rows of K / 2 bytes.
    const bool fp4 = in_dtype == GEMM_E2M1;
    const int64_t epu = fp4 ? 2 : 1;   // elements per copied unit
    const int64_t Ku = K / epu;
    lda /= epu;
    ldb /= epu;
    const int isz = fp4 ? 1 : elem_size(in_dtype);
    const int osz = elem_size(out_dtype);
    const bool has_c = beta != 0.0f;
    const bool f8 = is_f8(in_dtype) || fp4;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto round_up = [](int64_t x, int64_t m) { return (x + m - 1) / m * m; };
    const int64_t a_rows = transA ? Ku : M, a_cols = transA ? M : Ku;
    const int64_t b_rows = transB ? N : Ku, b_cols = transB ? Ku : N;
    // 8-bit operands end up K-major: A as [M, K] (transA2 = 0), B as [N, K] (transB2 = 1)
    const int transA2 = f8 ? 0 : transA;
    const int transB2 = f8 ? 1 : transB;
    const bool a_turn = transA2 != transA, b_turn = transB2 != transB;
    const bool a_ok = !a_turn && a16(A) && (lda * isz) % 16 == 0;
    const bool b_ok = !b_turn && a16(B) && (ldb * isz) % 16 == 0;
    const bool d_ok = a16(D) && (ldd * osz) % 16 == 0;
    const bool c_ok = !has_c || (a16(C) && (ldc * osz) % 16 == 0);
    const int64_t per16 = 16 / isz;   // elements per 16 bytes
    const int64_t a_rows2 = a_turn ? a_cols : a_rows, a_cols2 = a_turn ? a_rows : a_cols;
    const int64_t b_rows2 = b_turn ? b_cols : b_rows, b_cols2 = b_turn ? b_rows : b_cols;
    const int64_t lda2 = a_ok ? lda : round_up(a_cols2, per16);
    const int64_t ldb2 = b_ok ? ldb : round_up(b_cols2, per16);
    const int64_t ldd2 = d_ok ? ldd : round_up(N, 16 / osz);
    const int64_t a_bytes = a_ok ? 0 : round_up(a_rows2 * lda2 * isz, 256);
    const int64_t b_bytes = b_ok ? 0 : round_up(b_rows2 * ldb2 * isz, 256);
    const int64_t d_bytes = d_ok ? 0 : round_up(M * ldd2 * osz, 256);
    void* ws = nullptr;
    uint32_t epoch = 0;
    if (workspace_for(kWsRepack, dev, s, a_bytes + b_bytes + d_bytes, &ws, &epoch, may_grow) != GEMM_OK)
        return kNoWorkspace;
    char* w = static_cast<char*>(ws);
    const void* A2 = A;
    const void* B2 = B;
    void* D2 = D;
    const void* C2 = C;
    int64_t ldc2 = ldc;
    cudaError_t e = cudaSuccess;
    if (!a_ok) {
        A2 = w;
        e = a_turn ? gb300::launch_transpose2d(w, lda2, A, lda, a_rows, a_cols, isz, s)
                   : gb300::launch_copy2d(w, lda2, A, lda, a_rows, a_cols, isz, s);
        w += a_bytes;
    }
    if (e == cudaSuccess && !b_ok) {
        B2 = w;
        e = b_turn ? gb300::launch_transpose2d(w, ldb2, B, ldb, b_rows, b_cols, isz, s)
                   : gb300::launch_copy2d(w, ldb2, B, ldb, b_rows, b_cols, isz, s);
        w += b_bytes;
    }
    if (!d_ok) D2 = w;
    if (e == cudaSuccess && has_c && !(c_ok && C != D)) {
        if (!(c_ok && d_ok)) {   // (C == D, both aligned: already in place)
            e = gb300::launch_copy2d(D2, ldd2, C, ldc, M, N, osz, s);
            C2 = D2;
            ldc2 = ldd2;
        }
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    const int rc = SFA ? gemm_mx(D2, A2, B2, C2, SFA, SFB, M, N, K, lda2 * epu, ldb2 * epu, ldc2, ldd2, ld_sfa, ld_sfb,
                                 transA2, transB2, alpha, beta, in_dtype, out_dtype, s)
                       : gemm(D2, A2, B2, C2, M, N, K, lda2, ldb2, ldc2, ldd2, transA2, transB2, alpha, beta,
                              in_dtype, out_dtype, s);
    if (rc != GEMM_OK || d_ok) return rc;
    if (gb300::launch_copy2d(D, ldd, D2, ldd2, M, N, osz, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

int gb300::pdl_setting() {
    static const int on = [] {
        const char* v = std::getenv("GEMM_PDL");
        return (v && std::strcmp(v, "0") == 0) ? 0 : 1;
    }();
    return on;
}

extern "C" {

const char* gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED_DTYPE: return "GEMM_ERR_UNSUPPORTED_DTYPE";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
        case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS";
        case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
        case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE";
        case GEMM_ERR_UNSUPPORTED_LAYOUT: return "GEMM_ERR_UNSUPPORTED_LAYOUT";
        default: return "GEMM_ERR_UNKNOWN";
    }
}

int gemm_tile_coords(int tile, int num_m, int num_n, int group_m, int* m_blk, int* n_blk) {
    if (num_m < 1 || num_n < 1 || group_m < 1 || tile < 0 || !m_blk || !n_blk) return GEMM_ERR_INVALID_ARG;
    if ((int64_t)num_m * num_n > kMaxDim || tile >= num_m * num_n) return GEMM_ERR_INVALID_ARG;
    gb300::tile_coords(tile, num_m, num_n, group_m, m_blk, n_blk);
    return GEMM_OK;
}

int gemm_schedule_units(int num_tiles, int iters, int workers, int sk_tiles, int worker, int* out, int max_units) {
    if (num_tiles < 1 || iters < 1 || workers < 1 || sk_tiles < 0 || sk_tiles > num_tiles || worker < 0 ||
        worker >= workers || max_units < 0 || (max_units > 0 && !out))
        return GEMM_ERR_INVALID_ARG;
    const gb300::Schedule s{num_tiles, iters, workers, sk_tiles};
    gb300::UnitIter it;
    it.start(s, worker);
    gb300::WorkUnit u;
    int n = 0;
    while (it.next(s, worker, &u)) {
        if (n < max_units) {
            int* r = out + 6 * n;
            r[0] = u.tile;
            r[1] = u.kb;
            r[2] = u.ke;
            r[3] = u.sk;
            r[4] = u.ci;
            r[5] = u.nc;
        }
        ++n;
    }
    return n;
}

int gemm_plan(int64_t M, int64_t N, int64_t K, int num_sms, int64_t* out) {
    return gemm_plan_layout(M, N, K, 0, GEMM_F16, GEMM_F32, num_sms, out);
}

int gemm_plan_layout(int64_t M, int64_t N, int64_t K, int transB, int in_dtype, int out_dtype, int num_sms,
                     int64_t* out) {
    if (M < 1 || N < 1 || K < 0 || num_sms < 2 || !out || (transB != 0 && transB != 1)) return GEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_TOO_LARGE;
    if ((in_dtype != GEMM_F16 && in_dtype != GEMM_BF16 && !is_f8(in_dtype)) ||
        (out_dtype != GEMM_F32 && out_dtype != GEMM_F16 && out_dtype != GEMM_BF16))
        return GEMM_ERR_UNSUPPORTED_DTYPE;
    // 8-bit operands always reach the kernel K-major (repacked if needed)
    const int f8 = is_f8(in_dtype) ? 1 : 0;
    Plan pl = make_plan(M, N, K, num_sms, true, out_dtype, f8, 0, f8 ? 1 : transB);
    out[0] = pl.pair;
    out[1] = pl.tile_m;
    out[2] = pl.tile_n;
    out[3] = pl.num_tiles;
    out[4] = pl.grid;
    out[5] = pl.smem;
    out[6] = pl.epi_warps;
    out[7] = pl.stages;
    out[8] = pl.sk_tiles;
    out[9] = pl.ws_bytes;
    return GEMM_OK;
}

int gemm(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K, int64_t lda,
         int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float alpha, float beta, int in_dtype,
         int out_dtype, struct CUstream_st* stream) {
    int rc = validate(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, beta, in_dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;

    // ---- device ----
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_CUDA, "cudaGetDevice");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Inside a CUDA graph capture nothing may be allocated: the device set-up
    // (one allocation) must have happened before, and workspaces are used
    // only where they already exist (see below).
    const bool in_capture = capturing(s);
    if (in_capture && !device_ready(dev))
        return reject(GEMM_ERR_CUDA, "first call on this device inside a stream capture");
    DeviceState* ds = nullptr;
    if ((rc = device_state(dev, &ds)) != GEMM_OK) return reject(rc, "device set-up");
    const bool has_c = beta != 0.0f;
    if (K == 0) {
        GEMM_LOGF("M=%lld N=%lld K=0: epilogue-only kernel", (long long)M, (long long)N);
        return launch_k0_or_reject(out_dtype, D, C, M, N, ldc, ldd, alpha, beta, ds->num_sms, s);
    }
    const bool f8 = is_f8(in_dtype);
    const bool direct_ok =
        tma_layout_ok(D, A, B, C, K, lda, ldb, ldc, ldd, elem_size(in_dtype), elem_size(out_dtype), has_c) &&
        operand_majors_ok(in_dtype, transA, transB);
    Route route = route_for(direct_ok, f8, true, M, N, K);
    if (route == kRouteRepack) {
        GEMM_LOGF("M=%lld N=%lld K=%lld: layout the tcgen05 kernel cannot take as it is, repacked", (long long)M,
                  (long long)N, (long long)K);
        rc = gemm_repacked(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta, in_dtype, out_dtype,
                           dev, s, !in_capture);
        if (rc != kNoWorkspace) return rc == GEMM_OK ? GEMM_OK : reject(rc, "repacked call");
        route = f8 ? kRouteNone : kRouteSync;   // no workspace to be had
    }
    if (route == kRouteNone) return reject(GEMM_ERR_UNSUPPORTED_LAYOUT, "8-bit operands: no workspace for repacking");
    if (route == kRouteSync) {
        GEMM_LOGF("M=%lld N=%lld K=%lld trans=%d%d: mma.sync kernel (%s)", (long long)M, (long long)N, (long long)K,
                  transA, transB, direct_ok ? "small problem" : "layout not 16-byte aligned");
        return launch_sync_or_reject(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta, in_dtype,
                                     out_dtype, s);
    }

    Plan pl = make_plan(M, N, K, plan_sms(ds->num_sms), true, out_dtype, f8 ? 1 : 0, 0, transB);
    void* ws = nullptr;
    uint32_t epoch = 0;
    if (pl.sk_tiles > 0 && workspace_for(kWsStreamK, dev, s, pl.ws_bytes, &ws, &epoch, !in_capture) != GEMM_OK) {
        if (!in_capture) return reject(GEMM_ERR_CUDA, "stream-K workspace");
        pl = make_plan(M, N, K, plan_sms(ds->num_sms), false, out_dtype, f8 ? 1 : 0, 0, transB);   // whole tiles: no workspace
    }
    TcgenLaunch L;
    if ((rc = describe_tcgen05(&L, pl, D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
                               in_dtype, out_dtype)) != GEMM_OK)
        return reject(rc, "tensor maps");
    GemmParams& p = L.p;
    p.status = ds->d_status;
    p.skip_first_stage = skip_first_stage_setting();
    if (pl.sk_tiles > 0) {
        p.sk_tiles = pl.sk_tiles;
        p.ws_max_nc = pl.max_nc;
        p.ws_epoch = epoch;
        p.ws_counters = static_cast<uint32_t*>(ws);
        p.ws_partials = static_cast<char*>(ws) + ((int64_t)pl.sk_tiles * 2 * 4 + 255) / 256 * 256;
    }
    GEMM_LOGF("M=%lld N=%lld K=%lld trans=%d%d in=%d out=%d beta%s0: %s tiles %dx%d (%d), grid %d, smem %d, "
              "%d epilogue warps, %d stages, %d stream-K tiles (<= %d contributors)",
              (long long)M, (long long)N, (long long)K, transA, transB, in_dtype, out_dtype, has_c ? "!=" : "==",
              pl.pair ? "cta-pair" : "1-cta", pl.tile_m, pl.tile_n, pl.num_tiles, pl.grid, pl.smem, pl.epi_warps,
              pl.stages, pl.sk_tiles, pl.max_nc);
    return launch_described(L, s);
}

int gemm_mx(void* D, const void* A, const void* B, const void* C, const void* SFA, const void* SFB, int64_t M,
            int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int64_t ld_sfa, int64_t ld_sfb,
            int transA, int transB, float alpha, float beta, int in_dtype, int out_dtype,
            struct CUstream_st* stream) {
    const bool fp4 = in_dtype == GEMM_E2M1;
    if (!is_f8(in_dtype) && !fp4)
        return reject(GEMM_ERR_UNSUPPORTED_DTYPE, "block scaling needs E4M3 / E5M2 / E2M1 operands");
    // Packed 4-bit operands: K-major only (A [M, K], B [N, K]), whole bytes
    // per row (K and the leading dimensions even).  Validated as the byte
    // matrices they are: A [M, K / 2], B [N, K / 2].
    if (fp4 && (transA != 0 || transB != 1) && M > 0 && N > 0 && K > 0)
        return reject(GEMM_ERR_UNSUPPORTED_LAYOUT, "4-bit operands must be K-major (transA = 0, transB = 1)");
    if (fp4 && K > 0 && M > 0 && N > 0 && ((K | lda | ldb) & 1))
        return reject(GEMM_ERR_INVALID_ARG, "4-bit operands: K, lda and ldb must be even");
    const int64_t epu = fp4 ? 2 : 1;   // elements per byte of A and B
    const int vdt = fp4 ? GEMM_E4M3 : in_dtype;
    const int64_t lda_in = lda, ldb_in = ldb;   // the caller's strides (lda / ldb may be redirected below)
    int rc = validate(D, A, B, C, M, N, K / epu, lda / epu, ldb / epu, ldc, ldd, transA, transB, beta, vdt, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    if ((rc = validate_scales(D, SFA, SFB, M, N, K, ld_sfa, ld_sfb, ldd, out_dtype)) != GEMM_OK) return rc;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_CUDA, "cudaGetDevice");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool in_capture = capturing(s);
    if (in_capture && !device_ready(dev))
        return reject(GEMM_ERR_CUDA, "first call on this device inside a stream capture");
    DeviceState* ds = nullptr;
    if ((rc = device_state(dev, &ds)) != GEMM_OK) return reject(rc, "device set-up");
    const bool has_c = beta != 0.0f;
    if (K == 0) return launch_k0_or_reject(out_dtype, D, C, M, N, ldc, ldd, alpha, beta, ds->num_sms, s);
    // Packed 4-bit operands reach shared memory through TMA's 16U4_ALIGN16B
    // type, which wants 32-byte-aligned rows of a multiple of 128 elements;
    // the other layouts are copied below into rows of K rounded up to 128,
    // zero-padded.  D and C follow gemm()'s rules.
    auto a32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
    const bool fp4_ops_ok = !fp4 || (a32(A) && a32(B) && lda % 64 == 0 && ldb % 64 == 0 && K % 128 == 0);
    const bool direct_ok = fp4 ? tma_layout_ok(D, nullptr, nullptr, C, 0, 0, 0, ldc, ldd, 1, elem_size(out_dtype), has_c)
                               : tma_layout_ok(D, A, B, C, K, lda, ldb, ldc, ldd, elem_size(in_dtype),
                                               elem_size(out_dtype), has_c) &&
                                     operand_majors_ok(in_dtype, transA, transB);
    if (!direct_ok) {
        GEMM_LOGF("mx: M=%lld N=%lld K=%lld: layout the tcgen05 kernel cannot take as it is, repacked", (long long)M,
                  (long long)N, (long long)K);
        rc = gemm_repacked(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta, in_dtype, out_dtype,
                           dev, s, !in_capture, SFA, SFB, ld_sfa, ld_sfb);
        if (rc != kNoWorkspace) return rc == GEMM_OK ? GEMM_OK : reject(rc, "repacked call");
        return reject(GEMM_ERR_UNSUPPORTED_LAYOUT, "8-bit operands: no workspace for repacking");
    }

    // Every workspace is acquired before anything is enqueued, so a refusal
    // (for instance inside a stream capture, which cannot allocate) leaves
    // the stream as it was.
    Plan pl = make_plan(M, N, K, plan_sms(ds->num_sms), true, out_dtype, 1, 1);
    // The scales, rearranged into 512-byte chunks (gemm_sm103_mx.cu): one per
    // 128-K sub-block and 128-row group of A (each CTA of a pair has its
    // own), and (tile N / 128) per sub-block and N tile.
    const int64_t kblocks = (K + 31) / 32;
    const int64_t kchunks = (int64_t)pl.iters * (gb300::tcgen05_stage_k(pl.pair, 1, pl.epi_warps, pl.tile_n) / 128);
    const int64_t a_groups = (int64_t)pl.num_m * (pl.pair ? 2 : 1);
    const int sfb_chunks = (pl.tile_n + 127) / 128;
    const int64_t sfa_bytes = gb300::sf_tiles_bytes(128, a_groups, kchunks);
    const int64_t sfb_bytes = gb300::sf_tiles_bytes(pl.tile_n, pl.num_n, kchunks);
    void* sws = nullptr;
    uint32_t sepoch = 0;
    if (workspace_for(kWsScales, dev, s, sfa_bytes + sfb_bytes, &sws, &sepoch, !in_capture) != GEMM_OK)
        return reject(GEMM_ERR_CUDA, in_capture ? "scale workspace (a capture cannot allocate it; make one call of "
                                                  "at least this size on the stream first)"
                                                : "scale workspace");
    uint8_t* sfa_tiles = static_cast<uint8_t*>(sws);
    uint8_t* sfb_tiles = sfa_tiles + sfa_bytes;
    void* ws = nullptr;
    uint32_t epoch = 0;
    if (pl.sk_tiles > 0 && workspace_for(kWsStreamK, dev, s, pl.ws_bytes, &ws, &epoch, !in_capture) != GEMM_OK) {
        if (!in_capture) return reject(GEMM_ERR_CUDA, "stream-K workspace");
        pl = make_plan(M, N, K, plan_sms(ds->num_sms), false, out_dtype, 1, 1);   // whole tiles: no workspace
    }
    // 4-bit operands off TMA's 4-bit grid: copied into zero-padded rows of K
    // rounded up to 128 elements.
    int64_t k_map = K;   // the K extent of the operand tensor maps
    uint8_t* a2 = nullptr;
    uint8_t* b2 = nullptr;
    const int64_t kp = (K + 127) / 128 * 128;
    const int64_t a2_bytes = (M * (kp / 2) + 255) / 256 * 256;
    const int64_t b2_bytes = (N * (kp / 2) + 255) / 256 * 256;
    if (!fp4_ops_ok) {
        void* fws = nullptr;
        uint32_t fepoch = 0;
        if (workspace_for(kWsFp4, dev, s, a2_bytes + b2_bytes, &fws, &fepoch, !in_capture) != GEMM_OK)
            return reject(GEMM_ERR_CUDA, "4-bit operand workspace");
        a2 = static_cast<uint8_t*>(fws);
        b2 = a2 + a2_bytes;
    }
    const void* A_op = a2 ? a2 : A;
    const void* B_op = b2 ? b2 : B;
    if (a2) {
        lda = ldb = k_map = kp;
    }

    TcgenLaunch L;
    // (packed 4-bit operands: maps of k_map elements per row; 128 of them
    // fill a 128-byte shared-memory row, as 8-bit ones do.  The operands take
    // whole-stage boxes like the plain kernel's: 8192^3 MX E4M3 +1.7 to
    // +2.6 %, E2M1 +2.0 to +2.4 %, 4096^3 MX E5M2 beta = 1 +1.2 %; the scale
    // boxes stay per sub-block, merging them too gained nothing measurable.)
    if ((rc = describe_tcgen05(&L, pl, D, A_op, B_op, C, M, N, k_map, lda, ldb, ldc, ldd, transA, transB, alpha,
                               beta, in_dtype, out_dtype)) != GEMM_OK)
        return reject(rc, "tensor maps");
    GemmParams& p = L.p;
    p.K = (int32_t)K;
    p.num_k_blocks = pl.iters;
    // tcgen05 instruction descriptor, kind::mxf8f6f4: A / B format (bits 7-9,
    // 10-12: 0 = E4M3, 1 = E5M2, 5 = E2M1), both K-major (bits 15, 16 = 0), N >> 3
    // (bits 17-22), scale type UE8M0 (bit 23), M >> 4 (bits 24-28); the
    // kernel adds the scale-byte IDs of each K slice (bits 4-5 for B, 29-30
    // for A).  The accumulator is f32 by definition of the kind.
    const uint32_t fmt = fp4 ? 5u : in_dtype == GEMM_E5M2 ? 1u : 0u;
    p.idesc = (fmt << 7) | (fmt << 10) | (((uint32_t)pl.tile_n >> 3) << 17) | (1u << 23) |
              (((uint32_t)pl.tile_m >> 4) << 24);
    if ((rc = encode_sf(&L.sfa, sfa_tiles, sfa_bytes / 512, 1)) != GEMM_OK ||
        (rc = encode_sf(&L.sfb, sfb_tiles, sfb_bytes / 512, (uint32_t)sfb_chunks)) != GEMM_OK)
        return reject(rc, "scale tensor maps");
    p.sf_a_groups = (int32_t)a_groups;
    p.operands_packed4 = fp4 ? 1 : 0;
    L.mx = 1;
    p.status = ds->d_status;
    p.skip_first_stage = skip_first_stage_setting();
    if (pl.sk_tiles > 0) {
        p.sk_tiles = pl.sk_tiles;
        p.ws_max_nc = pl.max_nc;
        p.ws_epoch = epoch;
        p.ws_counters = static_cast<uint32_t*>(ws);
        p.ws_partials = static_cast<char*>(ws) + ((int64_t)pl.sk_tiles * 2 * 4 + 255) / 256 * 256;
    }
    // ---- enqueue: the 4-bit operand copies, the scale rearranging, the product ----
    cudaError_t e = cudaSuccess;
    if (a2) {
        GEMM_LOGF("mx: 4-bit operands copied into 32-byte-aligned rows of %lld elements", (long long)kp);
        if (cudaMemsetAsync(a2, 0, (size_t)(a2_bytes + b2_bytes), s) != cudaSuccess)
            e = cudaErrorUnknown;
        if (e == cudaSuccess) e = gb300::launch_copy2d(a2, kp / 2, A, lda_in / 2, M, K / 2, 1, s);
        if (e == cudaSuccess) e = gb300::launch_copy2d(b2, kp / 2, B, ldb_in / 2, N, K / 2, 1, s);
    }
    if (e == cudaSuccess)
        e = gb300::launch_sf_tiles(
            gb300::sf_job(sfa_tiles, static_cast<const uint8_t*>(SFA), ld_sfa, M, kblocks, 128, a_groups, kchunks),
            gb300::sf_job(sfb_tiles, static_cast<const uint8_t*>(SFB), ld_sfb, N, kblocks, pl.tile_n, pl.num_n, kchunks),
            s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_LAUNCH, cudaGetErrorString(e));
    }
    GEMM_LOGF("mx: M=%lld N=%lld K=%lld in=%d out=%d beta%s0: %s tiles %dx%d (%d), grid %d, smem %d, %d stages, "
              "%d stream-K tiles",
              (long long)M, (long long)N, (long long)K, in_dtype, out_dtype, has_c ? "!=" : "==",
              pl.pair ? "cta-pair" : "1-cta", pl.tile_m, pl.tile_n, pl.num_tiles, pl.grid, pl.smem, pl.stages,
              pl.sk_tiles);
    return launch_described(L, s);
}

int gemm_poll_device_error(struct CUstream_st* stream, int* info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    // The two records this device may have: gemm()'s (cudaMalloc'd at its
    // first call) and gemm_noalloc()'s (the static array).  Only records
    // whose set-up has succeeded are read; none is created here, so a
    // caller that never lets the library allocate can poll too.
    DeviceStatus* records[2] = {gemm_status_record(dev), noalloc_status_record(dev)};
    if (info) info[0] = info[1] = info[2] = info[3] = 0;
    for (DeviceStatus* rec : records) {
        if (rec == nullptr) continue;
        DeviceStatus st{};
        if (cudaMemcpy(&st, rec, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (st.code == 0) continue;
        if (info) {
            info[0] = st.code;
            info[1] = st.block;
            info[2] = st.site;
            info[3] = st.detail;
        }
        // Clear the record that is reported; a second one, if it also
        // holds an error, is reported by the next poll.
        if (cudaMemset(rec, 0, sizeof(DeviceStatus)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return st.code;
    }
    return GEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_noalloc(): the same computation for callers that must not allocate
// device memory.  Its set-up (once per device) only queries attributes, sets
// the kernels' shared-memory limit and looks up the static scratch's device
// address; each call then validates, encodes the TMA maps on the host
// stack and launches.  The kernel's status record is the static array's
// first 16 bytes: zero when the library is loaded, it keeps the first wait
// that gave up until gemm_poll_device_error() reads and clears it.  Nothing
// on this path calls cudaMalloc, cudaFree or any other allocating routine.

namespace {

struct NoAllocState {
    bool ready = false;                       // set-up done and succeeded
    int num_sms = 0;
    DeviceStatus* scratch_status = nullptr;   // device address of the static scratch
};

NoAllocState g_noalloc[kMaxDevices];

// The one-time set-up of `dev` (the current device).  Only a successful
// set-up is kept: after a failure the next call tries again.
int noalloc_device_state(int dev, NoAllocState** out) {
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    NoAllocState& st = g_noalloc[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0, status = GEMM_OK;
        void* scratch = nullptr;
        if (fail_setup_setting()) {
            status = GEMM_ERR_CUDA;
        } else if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            status = GEMM_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            status = GEMM_ERR_ARCH;
        } else if (gb300::prepare_kernels_on_current_device() != cudaSuccess) {
            status = GEMM_ERR_CUDA;
        } else if (gb300::noalloc_scratch_address(&scratch) != cudaSuccess || scratch == nullptr) {
            status = GEMM_ERR_CUDA;
        }
        if (status != GEMM_OK) {
            cudaGetLastError();
            return status;
        }
        st.num_sms = sms;
        st.scratch_status = static_cast<DeviceStatus*>(scratch);
        st.ready = true;
    }
    *out = &st;
    return GEMM_OK;
}

DeviceStatus* noalloc_status_record(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    return g_noalloc[dev].ready ? g_noalloc[dev].scratch_status : nullptr;
}

}  // namespace

extern "C" GEMM_API int gemm_noalloc(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N,
                                     int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA,
                                     int transB, float alpha, float beta, int in_dtype, int out_dtype,
                                     struct CUstream_st* stream) {
    int rc = validate(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, beta, in_dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    const bool has_c = beta != 0.0f;
    const bool f8 = is_f8(in_dtype);
    const bool direct_ok =
        tma_layout_ok(D, A, B, C, K, lda, ldb, ldc, ldd, elem_size(in_dtype), elem_size(out_dtype), has_c) &&
        operand_majors_ok(in_dtype, transA, transB);
    const Route route = K == 0 ? kRouteTcgen05 : route_for(direct_ok, f8, false, M, N, K);
    if (route == kRouteNone)   // decided on the host: nothing enqueued
        return reject(GEMM_ERR_UNSUPPORTED_LAYOUT, "8-bit operands must be K-major and 16-byte aligned here");
    // The only scratch is the 16-byte status record, whatever the sizes;
    // refuse anything that would not fit the static array.
    if ((int)sizeof(DeviceStatus) > gb300::noalloc_scratch_bytes())
        return reject(GEMM_ERR_TOO_LARGE, "scratch larger than the static array");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_CUDA, "cudaGetDevice");
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (capturing(s)) {   // the one-time set-up is not done inside a stream capture
        std::lock_guard<std::mutex> lock(g_mutex);
        if (dev < 0 || dev >= kMaxDevices || !g_noalloc[dev].ready)
            return reject(GEMM_ERR_CUDA, "first call on this device inside a stream capture");
    }
    NoAllocState* ns = nullptr;
    if ((rc = noalloc_device_state(dev, &ns)) != GEMM_OK) return reject(rc, "device set-up (no-alloc)");
    if (K == 0)   // epilogue-only kernel: no scratch at all
        return launch_k0_or_reject(out_dtype, D, C, M, N, ldc, ldd, alpha, beta, ns->num_sms, s);
    if (route == kRouteSync)   // needs no scratch either
        return launch_sync_or_reject(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta, in_dtype,
                                     out_dtype, s);
    const Plan pl = make_plan(M, N, K, plan_sms(ns->num_sms), false, out_dtype, f8 ? 1 : 0, 0, transB);   // no workspace: data-parallel
    TcgenLaunch L;
    if ((rc = describe_tcgen05(&L, pl, D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, alpha, beta,
                               in_dtype, out_dtype)) != GEMM_OK)
        return reject(rc, "tensor maps");
    // The status record keeps the first wait that gave up since the last
    // gemm_poll_device_error(), which reads and clears it; it is zero when
    // the library is loaded.
    L.p.status = ns->scratch_status;
    L.p.skip_first_stage = skip_first_stage_setting();
    GEMM_LOGF("no-alloc: M=%lld N=%lld K=%lld: %s tiles %dx%d (%d), grid %d", (long long)M, (long long)N,
              (long long)K, pl.pair ? "cta-pair" : "1-cta", pl.tile_m, pl.tile_n, pl.num_tiles, pl.grid);
    return launch_described(L, s);
}
