// attention_forward_run on host buffers: the heads are split into parts whose
// copies in and out overlap each other and the attention kernels.
//
// Part i's Q, K and V are copied into the caller's device workspace on one
// stream while part i-1 runs on the caller's stream and part i-2's O and
// log-sum-exp are copied back on a third. Every head is independent, so a part
// is simply a smaller batch handed to attention_forward_run at offset views of
// the workspace. Only the public entry point of attention.cu is used here.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "attention.h"
#include "host_env.h"

namespace {

constexpr int kParts = 8;
constexpr size_t kRegionAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t q, k, v, o, lse, total;      // byte offsets of the regions in the workspace
};

Layout layout_for(int64_t batch, int64_t sq, int64_t sk, int64_t d, int out_f32) {
    const size_t b = (size_t)batch;
    const size_t q_bytes = b * (size_t)sq * (size_t)d * 2;
    const size_t kv_bytes = b * (size_t)sk * (size_t)d * 2;
    const size_t o_bytes = b * (size_t)sq * (size_t)d * (out_f32 ? 4 : 2);
    const size_t lse_bytes = b * (size_t)sq * 4;
    Layout l;
    l.q = 0;
    l.k = round_up(l.q + q_bytes, kRegionAlign);
    l.v = round_up(l.k + kv_bytes, kRegionAlign);
    l.o = round_up(l.v + kv_bytes, kRegionAlign);
    l.lse = round_up(l.o + o_bytes, kRegionAlign);
    l.total = round_up(l.lse + lse_bytes, kRegionAlign);
    return l;
}

// Streams and events of one call, released when the call returns.
struct Pipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, out_done = nullptr, ev_in[kParts] = {}, ev_run[kParts] = {};
    cudaError_t init() {
        cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&out_done, cudaEventDisableTiming);
        for (int i = 0; i < kParts && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&ev_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_run[i], cudaEventDisableTiming);
        }
        return e;
    }
    ~Pipe() {
        if (in) cudaStreamDestroy(in);
        if (out) cudaStreamDestroy(out);
        if (start) cudaEventDestroy(start);
        if (out_done) cudaEventDestroy(out_done);
        for (int i = 0; i < kParts; ++i) {
            if (ev_in[i]) cudaEventDestroy(ev_in[i]);
            if (ev_run[i]) cudaEventDestroy(ev_run[i]);
        }
    }
};

}  // namespace

extern "C" size_t attention_forward_host_workspace_bytes(int64_t batch, int64_t sq, int64_t sk, int64_t d,
                                                        int out_f32) {
    if (batch <= 0 || sq <= 0 || sk <= 0 || d <= 0) return 0;
    return layout_for(batch, sq, sk, d, out_f32).total;
}

extern "C" gemm_status_t attention_forward_run_host(const void* Q, const void* K, const void* V, void* O, float* lse,
                                                    int64_t batch, int64_t sq, int64_t sk, int64_t d, float scale,
                                                    int out_f32, int cluster, int cta_group, int causal,
                                                    void* workspace, size_t workspace_bytes, void* stream_v) {
    if (batch < 0 || sq < 0 || sk < 0) return GEMM_ERR_INVALID_ARG;
    if (batch == 0 || sq == 0) return GEMM_OK;
    if (sk == 0 || batch >= (1ll << 31) || sq >= (1ll << 31) || sk >= (1ll << 31)) return GEMM_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || (cluster != 1 && cluster != 2 && cluster != 4) || (cta_group != 1 && cta_group != 2) ||
        (cta_group == 2 && (cluster != 2 || d != 128)))
        return GEMM_ERR_UNSUPPORTED;
    if (cluster > 1 && cta_group == 1 && dgc_host::world_is_multi_gpu()) return GEMM_ERR_UNSUPPORTED;   // multicast
    if (!Q || !K || !V || !O || !workspace) return GEMM_ERR_INVALID_ARG;
    const Layout l = layout_for(batch, sq, sk, d, out_f32);
    if (workspace_bytes < l.total) return GEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & (kRegionAlign - 1)) return GEMM_ERR_ALIGNMENT;

    // Parts of whole heads; a part's lse view must start 16-byte aligned, so with
    // sq not a multiple of 4 the part size is a multiple of 4 / gcd(sq, 4) heads.
    const int64_t quantum = sq % 4 == 0 ? 1 : (sq % 2 == 0 ? 2 : 4);
    int64_t step = (batch + kParts - 1) / kParts;
    step = (step + quantum - 1) / quantum * quantum;
    const int64_t parts = (batch + step - 1) / step;

    char* ws = static_cast<char*>(workspace);
    const size_t q_head = (size_t)sq * d * 2, kv_head = (size_t)sk * d * 2;
    const size_t o_head = (size_t)sq * d * (out_f32 ? 4 : 2), lse_head = (size_t)sq * 4;
    const char* hq = static_cast<const char*>(Q);
    const char* hk = static_cast<const char*>(K);
    const char* hv = static_cast<const char*>(V);
    char* ho = static_cast<char*>(O);
    char* hl = reinterpret_cast<char*>(lse);
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

    Pipe pipe;
    cudaError_t e = pipe.init();
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    gemm_status_t s = GEMM_OK;
    e = cudaEventRecord(pipe.start, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.in, pipe.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.out, pipe.start, 0);
    for (int64_t i = 0; i < parts && e == cudaSuccess; ++i) {
        const int64_t h0 = i * step, hb = std::min(batch, h0 + step) - h0;
        const size_t qo = (size_t)h0 * q_head, ko = (size_t)h0 * kv_head;
        const size_t oo = (size_t)h0 * o_head, lo = (size_t)h0 * lse_head;
        e = cudaMemcpyAsync(ws + l.q + qo, hq + qo, (size_t)hb * q_head, cudaMemcpyHostToDevice, pipe.in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ws + l.k + ko, hk + ko, (size_t)hb * kv_head, cudaMemcpyHostToDevice, pipe.in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ws + l.v + ko, hv + ko, (size_t)hb * kv_head, cudaMemcpyHostToDevice, pipe.in);
        if (e == cudaSuccess) e = cudaEventRecord(pipe.ev_in[i], pipe.in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, pipe.ev_in[i], 0);
        if (e != cudaSuccess) break;
        s = attention_forward_run(ws + l.q + qo, ws + l.k + ko, ws + l.v + ko, ws + l.o + oo,
                                  lse ? reinterpret_cast<float*>(ws + l.lse + lo) : nullptr, hb, sq, sk, d, scale,
                                  out_f32, cluster, cta_group, causal, stream_v);
        if (s != GEMM_OK) break;
        e = cudaEventRecord(pipe.ev_run[i], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(pipe.out, pipe.ev_run[i], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(ho + oo, ws + l.o + oo, (size_t)hb * o_head, cudaMemcpyDeviceToHost, pipe.out);
        if (e == cudaSuccess && lse)
            e = cudaMemcpyAsync(hl + lo, ws + l.lse + lo, (size_t)hb * lse_head, cudaMemcpyDeviceToHost, pipe.out);
    }
    if (e == cudaSuccess && s == GEMM_OK) {
        e = cudaEventRecord(pipe.out_done, pipe.out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, pipe.out_done, 0);
    }
    // Nothing may still touch the caller's host buffers once this returns.
    const cudaError_t e_in = cudaStreamSynchronize(pipe.in);
    const cudaError_t e_out = cudaStreamSynchronize(pipe.out);
    const cudaError_t e_s = cudaStreamSynchronize(stream);
    if (s != GEMM_OK) return s;
    if (e != cudaSuccess || e_in != cudaSuccess || e_out != cudaSuccess || e_s != cudaSuccess) return GEMM_ERR_CUDA;
    return attention_forward_query_status(stream_v);
}
