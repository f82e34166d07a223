// Host-side internals shared by the GEMM library's translation units (not part
// of the C ABI): the handle, the failure recorder, and the launch path that the
// host-buffer entry points (host_io.cu) call on their staging buffers.
#ifndef DGC_GEMM_INTERNAL_H
#define DGC_GEMM_INTERNAL_H

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "densegemm.h"

namespace dgc_host {

constexpr int kHostChunks = 8;   // most parts the host-buffer entry points split a problem into

// Records a formatted reason on `sink` (or, when null, for the calling thread)
// and returns `s`.
gemm_status_t fail(std::string* sink, gemm_status_t s, const char* fmt, ...);

}  // namespace dgc_host

struct gemm_handle_s {
    gemm_options_t opt;
    int device = 0;
    int sm_count = 0;
    unsigned int* d_status = nullptr;
    unsigned long long* d_clock = nullptr;   // clock probe: cycles, nanoseconds, CTAs
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::string err;
    // Host-buffer entry points: device staging for A, B and C (grown on demand),
    // streams for host-to-device and device-to-host copies, and the events that
    // order them against the caller's stream.
    void* stage_ptr[3] = {nullptr, nullptr, nullptr};
    size_t stage_cap[3] = {0, 0, 0};
    bool pipe_ready = false;
    cudaStream_t pipe_in = nullptr, pipe_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_whole = nullptr, ev_out_done = nullptr;
    cudaEvent_t ev_in[dgc_host::kHostChunks] = {}, ev_c[dgc_host::kHostChunks] = {};
    int64_t launches = 0;
    bool no_alloc = false;      // set on the stack handle of gemm_run_noalloc: never allocate
    bool status_cleared = false;// gemm_run_noalloc: the launch path cleared the static record (a GEMM kernel followed)
    float* workspace = nullptr; // stream-K partial slots
    unsigned int* flags = nullptr;
    size_t workspace_bytes = 0;
    size_t flag_count = 0;
    bool smem_set[2][2][2] = {};
    int occ_key[2][2][2][9];    // cached max active clusters per (BN, G, BK, cluster size)
};

namespace dgc_host {

// gemm_run_strided_batched on device pointers: validation, planning, tensor maps
// and the launch (batch = 1 is gemm_run).
gemm_status_t run_impl(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       int64_t strideA, const void* B, int64_t ldb, int64_t strideB, void* C, int64_t ldc,
                       int64_t strideC, int64_t batch, float alpha, float beta, void* stream);

}  // namespace dgc_host

#endif  // DGC_GEMM_INTERNAL_H
