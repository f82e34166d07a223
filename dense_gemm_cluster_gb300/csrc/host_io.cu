// Host-buffer entry points of the C ABI declared in include/densegemm.h:
// gemm_run_host and gemm_run_strided_batched_host copy the caller's host
// matrices through handle-owned device staging, in parts whose copies in, GEMMs
// and copies out overlap on three streams.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "gemm_internal.h"

using namespace dgc_host;

namespace {

gemm_status_t ensure_stage(gemm_handle_t h, int i, size_t bytes) {
    if (h->stage_cap[i] >= bytes) return GEMM_OK;
    if (h->stage_ptr[i]) cudaFree(h->stage_ptr[i]);
    h->stage_ptr[i] = nullptr;
    h->stage_cap[i] = 0;
    cudaError_t e = cudaMalloc(&h->stage_ptr[i], bytes);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "staging buffer: %s", cudaGetErrorString(e));
    h->stage_cap[i] = bytes;
    return GEMM_OK;
}

// gemm_run_host splits the problem along the larger of M and N into up to
// kHostChunks parts. The operand that every part needs is copied in whole first;
// then part i's slice of the other operand (and of C when beta != 0) is copied in
// on one stream while part i-1 computes on the caller's stream and part i-2's C
// is copied out on a third, so the copies in both directions overlap each other
// and the GEMMs. The part count is the one with the least modelled time: copies
// at the host link's rate, each part's GEMM as whole waves of tiles at a busy
// SM's rate, so parts stay large enough to fill the GPU.
constexpr int64_t kHostChunkAlign = 256;   // keeps every slice start 16-byte aligned
constexpr double kHostToDeviceBps = 200e9; // pinned copies over the GB300 host link, each way
constexpr double kDeviceToHostBps = 190e9;
constexpr double kTileFlopsPerSec = 9e12;  // one SM's rate on a 128 x block_n tile in a full wave
constexpr double kLaunchSec = 6e-6;        // host cost of one gemm_run (tensor maps and launch)

struct PartPlan {
    int64_t parts, step;
};

// Models the pipeline for each part count and returns the fastest split of the
// P-long dimension. `x_bytes_per_line` and `c_bytes_per_line` are the bytes one
// line of the split dimension adds to the copies in (sliced operand, plus C when
// read) and out; `whole_bytes` is the operand copied in whole.
static PartPlan choose_parts(int64_t P, int64_t other, int64_t K, int BN, bool along_m, int sm_count,
                             double whole_bytes, double x_bytes_per_line, double c_in_bytes_per_line,
                             double c_out_bytes_per_line) {
    PartPlan best{1, P};
    double best_t = 1e30;
    for (int64_t n = 1; n <= kHostChunks; ++n) {
        int64_t step = (P + n - 1) / n;
        step = (step + kHostChunkAlign - 1) / kHostChunkAlign * kHostChunkAlign;
        const int64_t parts = (P + step - 1) / step;
        if (parts != n) continue;
        double in_done = whole_bytes / kHostToDeviceBps, g_end = 0.0, d_end = 0.0;
        for (int64_t i = 0; i < parts; ++i) {
            const int64_t r = std::min(step, P - i * step);
            in_done += (double)r * (x_bytes_per_line + c_in_bytes_per_line) / kHostToDeviceBps;
            const int64_t tiles = along_m ? ((r + 127) / 128) * ((other + BN - 1) / BN)
                                          : ((other + 127) / 128) * ((r + BN - 1) / BN);
            const double waves = (double)((tiles + sm_count - 1) / sm_count);
            const double g = kLaunchSec + waves * 2.0 * 128.0 * BN * (double)K / kTileFlopsPerSec;
            g_end = std::max(in_done, g_end) + g;
            d_end = std::max(g_end, d_end) + (double)r * c_out_bytes_per_line / kDeviceToHostBps;
        }
        if (d_end < best_t * 0.98) {      // prefer fewer parts unless more save at least 2 %
            best_t = d_end;
            best = PartPlan{parts, step};
        }
    }
    return best;
}

// One matrix as stored: `outer` lines of `inner` elements, `ld` elements apart.
struct HostMat {
    const char* host;
    char* dev;
    int64_t outer, inner, ld;
    int esize;
};

// Copies lines [o0, o1) and elements [i0, i1) of each line, pitched on both
// sides so the padding between lines is never written.
static cudaError_t copy_block(const HostMat& m, int64_t o0, int64_t o1, int64_t i0, int64_t i1, bool to_device,
                              cudaStream_t s) {
    if (o1 <= o0 || i1 <= i0) return cudaSuccess;
    const size_t pitch = (size_t)m.ld * m.esize;
    const size_t off = (size_t)o0 * pitch + (size_t)i0 * m.esize;
    const size_t width = (size_t)(i1 - i0) * m.esize;
    const size_t lines = (size_t)(o1 - o0);
    char* dev = m.dev + off;
    char* host = const_cast<char*>(m.host) + off;
    if (width == pitch)
        return to_device ? cudaMemcpyAsync(dev, host, width * lines, cudaMemcpyHostToDevice, s)
                         : cudaMemcpyAsync(host, dev, width * lines, cudaMemcpyDeviceToHost, s);
    return to_device ? cudaMemcpy2DAsync(dev, pitch, host, pitch, width, lines, cudaMemcpyHostToDevice, s)
                     : cudaMemcpy2DAsync(host, pitch, dev, pitch, width, lines, cudaMemcpyDeviceToHost, s);
}

// Copies the slice [c0, c1) of the chunked dimension: the lines when that
// dimension is the matrix's outer one, else the same columns of every line.
static cudaError_t copy_slice(const HostMat& m, bool chunk_is_outer, int64_t c0, int64_t c1, bool to_device,
                              cudaStream_t s) {
    return chunk_is_outer ? copy_block(m, c0, c1, 0, m.inner, to_device, s)
                          : copy_block(m, 0, m.outer, c0, c1, to_device, s);
}

static gemm_status_t pipe_setup(gemm_handle_t h) {
    if (h->pipe_ready) return GEMM_OK;
    cudaError_t e = cudaStreamCreateWithFlags(&h->pipe_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->pipe_out, cudaStreamNonBlocking);
    cudaEvent_t* evs[3] = {&h->ev_start, &h->ev_whole, &h->ev_out_done};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    for (int i = 0; i < kHostChunks && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_c[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        // release what was created so a later call starts from nothing
        if (h->pipe_in) cudaStreamDestroy(h->pipe_in);
        if (h->pipe_out) cudaStreamDestroy(h->pipe_out);
        for (int i = 0; i < 3; ++i)
            if (*evs[i]) cudaEventDestroy(*evs[i]);
        for (int i = 0; i < kHostChunks; ++i) {
            if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
            if (h->ev_c[i]) cudaEventDestroy(h->ev_c[i]);
            h->ev_in[i] = h->ev_c[i] = nullptr;
        }
        h->pipe_in = h->pipe_out = nullptr;
        h->ev_start = h->ev_whole = h->ev_out_done = nullptr;
        return fail(&h->err, GEMM_ERR_CUDA, "copy pipeline set-up: %s", cudaGetErrorString(e));
    }
    h->pipe_ready = true;
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A,
                                       int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                                       float alpha, float beta, void* stream_v) {
    if (!h) return fail(nullptr, GEMM_ERR_INVALID_ARG, "null handle");
    if (M < 0 || N < 0 || K < 0) return fail(&h->err, GEMM_ERR_INVALID_ARG, "negative size");
    if (M == 0 || N == 0) return GEMM_OK;
    const gemm_options_t& o = h->opt;
    const int esc = o.out_type == GEMM_OUT_F32 ? 4 : 2;
    if (!C || (K > 0 && (!A || !B))) return fail(&h->err, GEMM_ERR_INVALID_ARG, "null host pointer");
    const bool a_row = o.layout_a == GEMM_ROW_MAJOR, b_row = o.layout_b == GEMM_ROW_MAJOR,
               c_row = o.layout_c == GEMM_ROW_MAJOR;
    // Leading dimensions are checked here (gemm_run checks them again) because the
    // staging sizes and the pitched copies depend on them.
    if (ldc < (c_row ? N : M) || (K > 0 && (lda < (a_row ? K : M) || ldb < (b_row ? N : K))))
        return fail(&h->err, GEMM_ERR_INVALID_ARG, "leading dimension smaller than the stored extent");
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    struct Restore {
        int d, p;
        ~Restore() { if (d != p) cudaSetDevice(p); }
    } restore{h->device, prev};
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

    HostMat a{static_cast<const char*>(A), nullptr, a_row ? M : K, a_row ? K : M, lda, 2};
    HostMat b{static_cast<const char*>(B), nullptr, b_row ? K : N, b_row ? N : K, ldb, 2};
    HostMat c{static_cast<const char*>(C), nullptr, c_row ? M : N, c_row ? N : M, ldc, esc};
    auto footprint = [](const HostMat& m) -> size_t {
        return m.outer == 0 || m.inner == 0 ? 0 : (size_t)((m.outer - 1) * m.ld + m.inner) * m.esize;
    };
    gemm_status_t s;
    if ((s = ensure_stage(h, 0, footprint(a) + 16)) != GEMM_OK) return s;
    if ((s = ensure_stage(h, 1, footprint(b) + 16)) != GEMM_OK) return s;
    if ((s = ensure_stage(h, 2, footprint(c) + 16)) != GEMM_OK) return s;
    if ((s = pipe_setup(h)) != GEMM_OK) return s;
    a.dev = static_cast<char*>(h->stage_ptr[0]);
    b.dev = static_cast<char*>(h->stage_ptr[1]);
    c.dev = static_cast<char*>(h->stage_ptr[2]);

    // Chunk the larger of M and N; the operand along the other one is copied whole.
    const bool along_m = M >= N;
    const int64_t P = along_m ? M : N, other = along_m ? N : M;
    PartPlan pp = choose_parts(P, other, K, o.block_n ? o.block_n : 256, along_m, h->sm_count,
                               (double)other * K * 2, (double)K * 2, beta != 0.0f ? (double)other * esc : 0.0,
                               (double)other * esc);
    if (o.host_parts > 0) {
        pp.step = ((P + o.host_parts - 1) / o.host_parts + kHostChunkAlign - 1) / kHostChunkAlign * kHostChunkAlign;
        pp.parts = (P + pp.step - 1) / pp.step;
    }
    const int64_t parts = pp.parts, step = pp.step;
    HostMat& x = along_m ? a : b;            // sliced operand
    HostMat& y = along_m ? b : a;            // whole operand
    const bool x_outer = along_m ? a_row : !b_row;   // the chunked dimension is x's line index
    const bool c_outer = along_m ? c_row : !c_row;

    cudaError_t e = cudaEventRecord(h->ev_start, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_in, h->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->ev_start, 0);
    if (e == cudaSuccess && K > 0) e = copy_block(y, 0, y.outer, 0, y.inner, true, h->pipe_in);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_whole, h->pipe_in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_whole, 0);
    for (int64_t i = 0; i < parts && e == cudaSuccess && s == GEMM_OK; ++i) {
        const int64_t c0 = i * step, c1 = std::min(P, c0 + step);
        if (K > 0) e = copy_slice(x, x_outer, c0, c1, true, h->pipe_in);
        if (e == cudaSuccess && beta != 0.0f) e = copy_slice(c, c_outer, c0, c1, true, h->pipe_in);
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[i], h->pipe_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_in[i], 0);
        if (e != cudaSuccess) break;
        // The part's operands as views into the staging buffers.
        const size_t xo = (size_t)c0 * (x_outer ? (size_t)x.ld : 1) * x.esize;
        const size_t co = (size_t)c0 * (c_outer ? (size_t)c.ld : 1) * c.esize;
        const int64_t mp = along_m ? c1 - c0 : M, np = along_m ? N : c1 - c0;
        const void* Ap = along_m ? (const void*)(a.dev + xo) : (const void*)a.dev;
        const void* Bp = along_m ? (const void*)b.dev : (const void*)(b.dev + xo);
        s = run_impl(h, mp, np, K, Ap, lda, 0, Bp, ldb, 0, c.dev + co, ldc, 0, 1, alpha, beta, stream_v);
        if (s != GEMM_OK) break;
        e = cudaEventRecord(h->ev_c[i], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->ev_c[i], 0);
        if (e == cudaSuccess) e = copy_slice(c, c_outer, c0, c1, false, h->pipe_out);
    }
    if (e == cudaSuccess && s == GEMM_OK) {
        e = cudaEventRecord(h->ev_out_done, h->pipe_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_out_done, 0);
    }
    // Whatever happened, nothing may still read or write the caller's host
    // buffers once this returns.
    const cudaError_t e_in = cudaStreamSynchronize(h->pipe_in);
    const cudaError_t e_out = cudaStreamSynchronize(h->pipe_out);
    const cudaError_t e_s = cudaStreamSynchronize(stream);
    if (s != GEMM_OK) return s;
    if (e == cudaSuccess) e = e_in != cudaSuccess ? e_in : (e_out != cudaSuccess ? e_out : e_s);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "host copy pipeline: %s", cudaGetErrorString(e));
    return GEMM_OK;
}

// gemm_run_strided_batched on host buffers: the batch is split into parts of
// whole products, pipelined like gemm_run_host's parts. An operand with stride 0
// (one matrix for every product) is copied once, first.
extern "C" gemm_status_t gemm_run_strided_batched_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                                       const void* A, int64_t lda, int64_t strideA, const void* B,
                                                       int64_t ldb, int64_t strideB, void* C, int64_t ldc,
                                                       int64_t strideC, int64_t batch, float alpha, float beta,
                                                       void* stream_v) {
    if (!h) return fail(nullptr, GEMM_ERR_INVALID_ARG, "null handle");
    if (M < 0 || N < 0 || K < 0 || batch < 0) return fail(&h->err, GEMM_ERR_INVALID_ARG, "negative size");
    if (M == 0 || N == 0 || batch == 0) return GEMM_OK;
    if (batch == 1) return gemm_run_host(h, M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, stream_v);
    const gemm_options_t& o = h->opt;
    const int esc = o.out_type == GEMM_OUT_F32 ? 4 : 2;
    if (!C || (K > 0 && (!A || !B))) return fail(&h->err, GEMM_ERR_INVALID_ARG, "null host pointer");
    const bool a_row = o.layout_a == GEMM_ROW_MAJOR, b_row = o.layout_b == GEMM_ROW_MAJOR,
               c_row = o.layout_c == GEMM_ROW_MAJOR;
    if (ldc < (c_row ? N : M) || (K > 0 && (lda < (a_row ? K : M) || ldb < (b_row ? N : K))))
        return fail(&h->err, GEMM_ERR_INVALID_ARG, "leading dimension smaller than the stored extent");
    HostMat a{static_cast<const char*>(A), nullptr, a_row ? M : K, a_row ? K : M, lda, 2};
    HostMat b{static_cast<const char*>(B), nullptr, b_row ? K : N, b_row ? N : K, ldb, 2};
    HostMat c{static_cast<const char*>(C), nullptr, c_row ? M : N, c_row ? N : M, ldc, esc};
    auto fp = [](const HostMat& m) -> int64_t { return m.outer == 0 || m.inner == 0 ? 0 : (m.outer - 1) * m.ld + m.inner; };
    if (strideC < c.outer * ldc ||
        (K > 0 && (strideA < 0 || strideB < 0 || (strideA != 0 && strideA < a.outer * lda) ||
                   (strideB != 0 && strideB < b.outer * ldb))))
        return fail(&h->err, GEMM_ERR_INVALID_ARG,
                    "strides must keep the matrices apart (A and B may also use 0: one matrix for every product)");
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    struct Restore {
        int d, p;
        ~Restore() { if (d != p) cudaSetDevice(p); }
    } restore{h->device, prev};
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const int64_t a_span = K > 0 ? (batch - 1) * strideA + fp(a) : 0;
    const int64_t b_span = K > 0 ? (batch - 1) * strideB + fp(b) : 0;
    const int64_t c_span = (batch - 1) * strideC + fp(c);
    gemm_status_t s;
    if ((s = ensure_stage(h, 0, (size_t)a_span * 2 + 16)) != GEMM_OK) return s;
    if ((s = ensure_stage(h, 1, (size_t)b_span * 2 + 16)) != GEMM_OK) return s;
    if ((s = ensure_stage(h, 2, (size_t)c_span * esc + 16)) != GEMM_OK) return s;
    if ((s = pipe_setup(h)) != GEMM_OK) return s;
    char* da = static_cast<char*>(h->stage_ptr[0]);
    char* db = static_cast<char*>(h->stage_ptr[1]);
    char* dc = static_cast<char*>(h->stage_ptr[2]);
    const char* ha = static_cast<const char*>(A);
    const char* hb = static_cast<const char*>(B);
    char* hc = static_cast<char*>(C);

    const int64_t want = o.host_parts > 0 ? o.host_parts : kHostChunks;
    const int64_t step = (batch + std::min<int64_t>(want, batch) - 1) / std::min<int64_t>(want, batch);
    const int64_t parts = (batch + step - 1) / step;
    const bool a_whole = K > 0 && strideA == 0;         // one A for every product: copy it once
    const bool b_whole = K > 0 && strideB == 0;
    const bool c_dense = ldc == c.inner && strideC == fp(c);
    // Bytes [first line of batch b0, end of batch b1 - 1) of an operand with stride st.
    auto span_copy = [](char* dev, const char* host, int64_t st, int64_t foot, int esize, int64_t b0, int64_t b1,
                        bool to_device, cudaStream_t cs) -> cudaError_t {
        const size_t off = (size_t)(b0 * st) * esize;
        const size_t bytes = (size_t)((b1 - 1 - b0) * st + foot) * esize;
        return to_device ? cudaMemcpyAsync(dev + off, host + off, bytes, cudaMemcpyHostToDevice, cs)
                         : cudaMemcpyAsync(const_cast<char*>(host) + off, dev + off, bytes, cudaMemcpyDeviceToHost, cs);
    };

    cudaError_t e = cudaEventRecord(h->ev_start, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_in, h->ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->ev_start, 0);
    if (e == cudaSuccess && a_whole) e = span_copy(da, ha, strideA, fp(a), 2, 0, batch, true, h->pipe_in);
    if (e == cudaSuccess && b_whole) e = span_copy(db, hb, strideB, fp(b), 2, 0, batch, true, h->pipe_in);
    for (int64_t i = 0; i < parts && e == cudaSuccess && s == GEMM_OK; ++i) {
        const int64_t b0 = i * step, b1 = std::min(batch, b0 + step);
        if (K > 0 && !a_whole) e = span_copy(da, ha, strideA, fp(a), 2, b0, b1, true, h->pipe_in);
        if (e == cudaSuccess && K > 0 && !b_whole) e = span_copy(db, hb, strideB, fp(b), 2, b0, b1, true, h->pipe_in);
        if (e == cudaSuccess && beta != 0.0f) e = span_copy(dc, hc, strideC, fp(c), esc, b0, b1, true, h->pipe_in);
        if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[i], h->pipe_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_in[i], 0);
        if (e != cudaSuccess) break;
        s = run_impl(h, M, N, K, da + (size_t)(b0 * strideA) * 2, lda, strideA, db + (size_t)(b0 * strideB) * 2, ldb,
                     strideB, dc + (size_t)(b0 * strideC) * esc, ldc, strideC, b1 - b0, alpha, beta, stream_v);
        if (s != GEMM_OK) break;
        e = cudaEventRecord(h->ev_c[i], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->pipe_out, h->ev_c[i], 0);
        if (c_dense) {
            if (e == cudaSuccess) e = span_copy(dc, hc, strideC, fp(c), esc, b0, b1, false, h->pipe_out);
        } else {
            // Padding between lines or batches stays untouched on the host.
            for (int64_t bb = b0; bb < b1 && e == cudaSuccess; ++bb) {
                const size_t off = (size_t)(bb * strideC) * esc;
                HostMat cb{hc + off, dc + off, c.outer, c.inner, ldc, esc};
                e = copy_block(cb, 0, c.outer, 0, c.inner, false, h->pipe_out);
            }
        }
    }
    if (e == cudaSuccess && s == GEMM_OK) {
        e = cudaEventRecord(h->ev_out_done, h->pipe_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, h->ev_out_done, 0);
    }
    const cudaError_t e_in = cudaStreamSynchronize(h->pipe_in);
    const cudaError_t e_out = cudaStreamSynchronize(h->pipe_out);
    const cudaError_t e_s = cudaStreamSynchronize(stream);
    if (s != GEMM_OK) return s;
    if (e == cudaSuccess) e = e_in != cudaSuccess ? e_in : (e_out != cudaSuccess ? e_out : e_s);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "host copy pipeline: %s", cudaGetErrorString(e));
    return GEMM_OK;
}
