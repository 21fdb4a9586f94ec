// gemm_host(): D = alpha * op(A) @ op(B) + beta * C with A, B, C, D in host
// memory (declared in include/gemm_gb300.h).
//
// The product runs on the device through gemm(); this file is the runtime
// around it: device staging buffers per (device, stream), and a pipeline
// over row panels of D on three streams, so that the host->device copies of
// later panels, the products of earlier ones and the device->host copies of
// finished ones overlap:
//
//   copy-in stream   B0 | A0 C0 | B1 | B2 | B3 | A1 C1 | A2 C2 | ...
//   caller's stream      | D00 | D01 | D02 | D03 |  gemm(panel 1) | ...
//   copy-out stream            | D00 | D01 | D02 | D03 |  D1  | ...
//
// A row panel of D needs all of B and its own rows of A (for transA = 1,
// its columns of the stored A, a strided copy) and C.  The first panel is
// computed and copied out in column blocks, each as soon as its block of B
// is in, so the copy-out stream starts long before all of B has crossed
// the host link.  The staging buffers have 16-byte-aligned row strides, so
// gemm() runs the tcgen05 kernel on them directly.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/gemm_gb300.h"

namespace {

constexpr int kMaxPanels = 16;
constexpr int kFirstBlocks = 4;   // column blocks of the first panel (N >= 1024)
constexpr int64_t kMaxDim = 2147483647;

int elem_bytes(int dtype) {
    if (dtype == GEMM_F32) return 4;
    if (dtype == GEMM_F16 || dtype == GEMM_BF16) return 2;
    if (dtype == GEMM_E4M3 || dtype == GEMM_E5M2) return 1;
    return 0;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Row panels of D: at most kMaxPanels, each a multiple of 256 rows (the
// CTA-pair tile height) and at least 1024 rows, so that every panel still
// fills the GPU with tiles.
int64_t panel_rows(int64_t M) {
    int64_t rows = std::max<int64_t>(1024, (M + kMaxPanels - 1) / kMaxPanels);
    return std::min(round_up(rows, 256), M);
}

// Staging buffers and streams of one (device, caller stream) pair.  Calls
// on one caller stream run in its order and share them; the events order a
// call's copies after the previous call's use of the same buffers.
struct Pipe {
    int dev = -1;
    cudaStream_t user = nullptr;
    cudaStream_t in = nullptr;    // host -> device copies
    cudaStream_t out = nullptr;   // device -> host copies
    cudaEvent_t loaded[kMaxPanels] = {};     // panel p's A (and C) are on the device
    cudaEvent_t computed[kMaxPanels] = {};   // panel p's D is on the device
    cudaEvent_t b_loaded[kFirstBlocks] = {};    // column block j of B is on the device
    cudaEvent_t b_computed[kFirstBlocks] = {};  // column block j of the first panel's D is on the device
    cudaEvent_t entry = nullptr;             // this call's place in the caller's stream
    cudaEvent_t copied_in = nullptr;         // the copy-in stream's work so far (failed calls)
    cudaEvent_t copied_out = nullptr;        // this call's D is on the host
    char* buf = nullptr;
    int64_t bytes = 0;
    bool captured = false;   // a CUDA graph captured copies into `buf`
    bool ready = false;
};

std::mutex g_mutex;
std::vector<Pipe*> g_pipes;
std::vector<char*> g_retired;   // replaced staging that captured graphs may still use

// True while `s` is being captured into a CUDA graph: nothing may be
// created or allocated then.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

int pipe_for(int dev, cudaStream_t user, bool may_create, Pipe** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (Pipe* p : g_pipes)
        if (p->dev == dev && p->user == user) {
            *out = p;
            return p->ready ? GEMM_OK : GEMM_ERR_CUDA;
        }
    if (!may_create) return GEMM_ERR_CUDA;
    Pipe* p = new Pipe;
    p->dev = dev;
    p->user = user;
    bool ok = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->entry, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->copied_in, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&p->copied_out, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxPanels; ++i)
        ok = cudaEventCreateWithFlags(&p->loaded[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->computed[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kFirstBlocks; ++i)
        ok = cudaEventCreateWithFlags(&p->b_loaded[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->b_computed[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) cudaGetLastError();
    p->ready = ok;
    g_pipes.push_back(p);   // kept until the process exits, like the device workspaces
    *out = p;
    return ok ? GEMM_OK : GEMM_ERR_CUDA;
}

// Grows the pipe's staging buffer.  Freeing the old one synchronises the
// device, so no copy or product still uses it; one that a captured graph
// has used is kept instead (until the process exits), since replays of
// that graph keep using its address.  `may_grow` false: inside a capture.
int ensure_buffer(Pipe* p, int64_t bytes, bool may_grow) {
    if (p->bytes >= bytes) {
        if (!may_grow) p->captured = true;
        return GEMM_OK;
    }
    if (!may_grow) return GEMM_ERR_CUDA;
    if (p->buf && p->captured) {
        std::lock_guard<std::mutex> lock(g_mutex);
        g_retired.push_back(p->buf);
    } else if (p->buf && cudaFree(p->buf) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    p->buf = nullptr;
    p->bytes = 0;
    p->captured = false;
    if (cudaMalloc(&p->buf, (size_t)bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    p->bytes = bytes;
    return GEMM_OK;
}

bool overlaps(const void* p, int64_t rows, int64_t cols, int64_t ld, int esz, const void* q, int64_t qrows,
              int64_t qcols, int64_t qld, int qesz) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
    const uintptr_t a1 = a0 + (uintptr_t)(((rows - 1) * ld + cols) * esz);
    const uintptr_t b1 = b0 + (uintptr_t)(((qrows - 1) * qld + qcols) * qesz);
    return a0 < b1 && b0 < a1;
}

// The host-side argument rules (the device-side ones are gemm()'s, which
// checks the staging layouts again).
int validate_host(const void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA, int transB, float beta,
                  int in_dtype, int out_dtype) {
    const int isz = elem_bytes(in_dtype), osz = elem_bytes(out_dtype);
    if (isz == 0 || isz == 4) return GEMM_ERR_UNSUPPORTED_DTYPE;
    if (osz == 0 || osz == 1) return GEMM_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_TOO_LARGE;
    const bool has_c = beta != 0.0f;
    if (!D || ldd < N) return GEMM_ERR_INVALID_ARG;
    if (has_c && (!C || ldc < N)) return GEMM_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B || lda < (transA ? M : K) || ldb < (transB ? K : N))) return GEMM_ERR_INVALID_ARG;
    const uintptr_t align = reinterpret_cast<uintptr_t>(D) | (has_c ? reinterpret_cast<uintptr_t>(C) : 0);
    if (align & (uintptr_t)(osz - 1)) return GEMM_ERR_MISALIGNED;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & (uintptr_t)(isz - 1)))
        return GEMM_ERR_MISALIGNED;
    if (K > 0 && (overlaps(D, M, N, ldd, osz, A, transA ? K : M, transA ? M : K, lda, isz) ||
                  overlaps(D, M, N, ldd, osz, B, transB ? N : K, transB ? K : N, ldb, isz)))
        return GEMM_ERR_ALIAS;
    if (has_c && C != D && overlaps(D, M, N, ldd, osz, C, M, N, ldc, osz)) return GEMM_ERR_ALIAS;
    if (has_c && C == D && ldc != ldd) return GEMM_ERR_ALIAS;
    return GEMM_OK;
}

int copy_error() {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
}

// A call that fails part-way, after some copies were enqueued on the side
// streams: the caller's stream is made to wait for them all the same, so
// that they stay inside "the stream has completed this call" (the host
// buffers must stay unchanged until then) and the next call's copies into
// the staging buffers cannot overtake them.
int fail_joined(Pipe* p, cudaStream_t user, int rc) {
    cudaGetLastError();
    if (cudaEventRecord(p->copied_in, p->in) == cudaSuccess) cudaStreamWaitEvent(user, p->copied_in, 0);
    if (cudaEventRecord(p->copied_out, p->out) == cudaSuccess) cudaStreamWaitEvent(user, p->copied_out, 0);
    cudaGetLastError();
    return rc;
}

}  // namespace

extern "C" GEMM_API int gemm_host(void* D, const void* A, const void* B, const void* C, int64_t M, int64_t N,
                                  int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t ldd, int transA,
                                  int transB, float alpha, float beta, int in_dtype, int out_dtype,
                                  struct CUstream_st* stream) {
    int rc = validate_host(D, A, B, C, M, N, K, lda, ldb, ldc, ldd, transA, transB, beta, in_dtype, out_dtype);
    if (rc != GEMM_OK || M == 0 || N == 0) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return copy_error();
    cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
    // Inside a CUDA graph capture the staging streams and buffers must exist
    // already (from an earlier call on this stream with at least these sizes).
    const bool may_allocate = !capturing(user);
    Pipe* p = nullptr;
    if ((rc = pipe_for(dev, user, may_allocate, &p)) != GEMM_OK) return rc;

    const bool has_c = beta != 0.0f;
    const int isz = elem_bytes(in_dtype), osz = elem_bytes(out_dtype);
    // staging layouts: rows padded to 16 bytes, each block 256-byte aligned
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    const int64_t lda_d = round_up(std::max<int64_t>(a_cols, 1), 16 / isz);
    const int64_t ldb_d = round_up(std::max<int64_t>(b_cols, 1), 16 / isz);
    const int64_t ldo_d = round_up(N, 16 / osz);   // C and D
    const int64_t a_bytes = round_up(a_rows * lda_d * isz, 256);
    const int64_t b_bytes = round_up(b_rows * ldb_d * isz, 256);
    const int64_t o_bytes = round_up(M * ldo_d * osz, 256);
    if ((rc = ensure_buffer(p, a_bytes + b_bytes + o_bytes * (has_c ? 2 : 1), may_allocate)) != GEMM_OK) return rc;
    char* dA = p->buf;
    char* dB = dA + a_bytes;
    char* dD = dB + b_bytes;
    char* dC = dD + o_bytes;

    // Stream order: the copies start after everything enqueued on the
    // caller's stream so far, which includes the previous call's copy-out
    // (see the end of this function), so the staging buffers are free.
    if (cudaEventRecord(p->entry, user) != cudaSuccess || cudaStreamWaitEvent(p->in, p->entry, 0) != cudaSuccess)
        return copy_error();
    const int64_t rows = panel_rows(M);
    const int panels = (int)((M + rows - 1) / rows);
    // columns [n0, n0 + nc) of op(B): a column block of the stored [K, N] B
    // (transB = 0), or a row block of the stored [N, K] B (transB = 1)
    const int64_t bcols = (N >= 1024 && K > 0) ? round_up((N + kFirstBlocks - 1) / kFirstBlocks, 256) : N;
    const int blocks = (int)((N + bcols - 1) / bcols);
    auto copy_b = [&](int64_t n0, int64_t nc) {
        if (transB)
            return cudaMemcpy2DAsync(dB + n0 * ldb_d * isz, ldb_d * isz, static_cast<const char*>(B) + n0 * ldb * isz,
                                     ldb * isz, K * isz, nc, cudaMemcpyHostToDevice, p->in);
        return cudaMemcpy2DAsync(dB + n0 * isz, ldb_d * isz, static_cast<const char*>(B) + n0 * isz, ldb * isz,
                                 nc * isz, K, cudaMemcpyHostToDevice, p->in);
    };
    auto b_block = [&](int64_t n0) -> const void* {
        return K > 0 ? static_cast<const void*>(dB + (transB ? n0 * ldb_d : n0) * isz) : nullptr;
    };
    // the rows of op(A) and of C of panel q, then its "loaded" event
    auto copy_panel_inputs = [&](int q) {
        const int64_t m0 = q * rows, mr = std::min(rows, M - m0);
        // rows m0.. of A, or columns m0.. of the stored [K, M] A
        const char* a_src = static_cast<const char*>(A) + (transA ? m0 : m0 * lda) * isz;
        char* a_dst = dA + (transA ? m0 : m0 * lda_d) * isz;
        if (K > 0 && cudaMemcpy2DAsync(a_dst, lda_d * isz, a_src, lda * isz, (transA ? mr : K) * isz,
                                       transA ? K : mr, cudaMemcpyHostToDevice, p->in) != cudaSuccess)
            return false;
        if (has_c && cudaMemcpy2DAsync(dC + m0 * ldo_d * osz, ldo_d * osz,
                                       static_cast<const char*>(C) + m0 * ldc * osz, ldc * osz, N * osz, mr,
                                       cudaMemcpyHostToDevice, p->in) != cudaSuccess)
            return false;
        return cudaEventRecord(p->loaded[q], p->in) == cudaSuccess;
    };
    // D[m0.., n0..] of the panel / block on the caller's stream, then its copy-out
    auto compute_and_return = [&](int q, int64_t n0, int64_t nc, cudaEvent_t inputs, cudaEvent_t done) {
        const int64_t m0 = q * rows, mr = std::min(rows, M - m0);
        if (cudaStreamWaitEvent(user, inputs, 0) != cudaSuccess) return copy_error();
        const void* a_panel = K > 0 ? static_cast<const void*>(dA + (transA ? m0 : m0 * lda_d) * isz) : nullptr;
        const int64_t o = (m0 * ldo_d + n0) * osz;
        int r = gemm(dD + o, a_panel, b_block(n0), has_c ? dC + o : nullptr, mr, nc, K, lda_d, ldb_d, ldo_d, ldo_d,
                     transA, transB, alpha, beta, in_dtype, out_dtype, stream);
        if (r != GEMM_OK) return r;
        if (cudaEventRecord(done, user) != cudaSuccess || cudaStreamWaitEvent(p->out, done, 0) != cudaSuccess ||
            cudaMemcpy2DAsync(static_cast<char*>(D) + (m0 * ldd + n0) * osz, ldd * osz, dD + o, ldo_d * osz,
                              nc * osz, mr, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
            return copy_error();
        return (int)GEMM_OK;
    };

    auto enqueue = [&]() -> int {
        // copy-in: B's first column block, the first panel's A and C, B's other blocks
        if (K > 0 && copy_b(0, std::min(bcols, N)) != cudaSuccess) return copy_error();
        if (!copy_panel_inputs(0)) return copy_error();
        for (int j = 1; j < blocks; ++j) {
            const int64_t n0 = j * bcols;
            if (copy_b(n0, std::min(bcols, N - n0)) != cudaSuccess ||
                cudaEventRecord(p->b_loaded[j], p->in) != cudaSuccess)
                return copy_error();
        }
        // the first panel, block by block
        int r;
        for (int j = 0; j < blocks; ++j) {
            const int64_t n0 = j * bcols;
            if ((r = compute_and_return(0, n0, std::min(bcols, N - n0), j == 0 ? p->loaded[0] : p->b_loaded[j],
                                        p->b_computed[j])) != GEMM_OK)
                return r;
        }
        // the other panels, whole
        for (int q = 1; q < panels; ++q) {
            if (!copy_panel_inputs(q)) return copy_error();
            if ((r = compute_and_return(q, 0, N, p->loaded[q], p->computed[q])) != GEMM_OK) return r;
        }
        // D is on the host when the caller's stream reaches this point.
        if (cudaEventRecord(p->copied_out, p->out) != cudaSuccess ||
            cudaStreamWaitEvent(user, p->copied_out, 0) != cudaSuccess)
            return copy_error();
        return GEMM_OK;
    };
    if ((rc = enqueue()) != GEMM_OK) return fail_joined(p, user, rc);
    return GEMM_OK;
}
