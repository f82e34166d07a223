// Host side of the C ABI declared in include/densegemm.h: option and argument
// validation, launch planning, TMA descriptor encoding, and the persistent
// cluster launch (the host-buffer entry points are in host_io.cu) ("Clusters, distributed shared memory & cluster launch
// control", section "Thread-block clusters": the cluster shape travels as a
// launch attribute of cudaLaunchKernelEx).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "densegemm.h"
#include "gemm_internal.h"
#include "host_env.h"
#include "gemm_kernel.cuh"

namespace dgc_host {

thread_local std::string g_thread_error;

gemm_status_t fail(std::string* sink, gemm_status_t s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    (sink ? *sink : g_thread_error) = buf;
    return s;
}

}  // namespace dgc_host

using namespace dgc_host;

namespace {

constexpr int kMaxSmemPerCta = 232448;        // 227 KB opt-in shared memory per block on sm_103
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// The clock probe's counters: three per SM slot.
constexpr size_t kClockBytes = 3 * dgc::CLOCK_PROBE_SLOTS * sizeof(unsigned long long);
constexpr int64_t kMinSplitBlocks = 16;         // k-blocks per cluster before a sub-wave problem is split wider
constexpr double kMinTailUs = 4.0;              // saved last-wave time worth a stream-K split
constexpr double kFlopPerUsPerSm = 1.5e9 / 152; // per-SM tensor rate for that estimate (1.5 PFLOP/s over 152 SMs)

bool pow2_le8(int v) { return v == 1 || v == 2 || v == 4 || v == 8; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One operand as the kernel sees it: a 3-D tensor (inner, outer, batch).
struct Operand {
    const void* ptr;
    int64_t ld;       // elements between consecutive outer indices
    int64_t stride;   // elements between batches
    bool mn_major;    // inner index runs along M (A) / N (B) rather than K
};

struct Resolved {
    gemm_plan_t pub;
    int64_t M, N, K;         // problem as launched (after the C^T transpose)
    int mcast_a, mcast_b;
    bool a_mn, b_mn;
    int out_f32;
};

// Everything gemm_run decides before touching the GPU.
gemm_status_t resolve(const gemm_options_t& o, int64_t M, int64_t N, int64_t K, int64_t batch,
                      int sm_count, Resolved& r, std::string* err) {
    if (o.mode != GEMM_MODE_UNICAST && o.mode != GEMM_MODE_MCAST)
        return fail(err, GEMM_ERR_INVALID_ARG, "mode must be GEMM_MODE_UNICAST or GEMM_MODE_MCAST");
    if ((o.layout_a | o.layout_b | o.layout_c) & ~1)
        return fail(err, GEMM_ERR_INVALID_ARG, "layouts must be GEMM_ROW_MAJOR or GEMM_COL_MAJOR");
    if (o.out_type != GEMM_OUT_BF16 && o.out_type != GEMM_OUT_F32)
        return fail(err, GEMM_ERR_INVALID_ARG, "out_type must be GEMM_OUT_BF16 or GEMM_OUT_F32");
    if (o.cta_group < 0 || o.cta_group > 2)
        return fail(err, GEMM_ERR_UNSUPPORTED, "cta_group must be 0 (auto), 1 or 2");
    if (!pow2_le8(o.cluster_m) || !pow2_le8(o.cluster_n) || o.cluster_m * o.cluster_n > 8)
        return fail(err, GEMM_ERR_UNSUPPORTED, "cluster %dx%d: each extent 1/2/4/8 and at most 8 CTAs",
                    o.cluster_m, o.cluster_n);
    if (o.block_n != 0 && o.block_n != 128 && o.block_n != 256)
        return fail(err, GEMM_ERR_UNSUPPORTED, "block_n must be 0, 128 or 256");
    if (o.block_k != 0 && o.block_k != 64 && o.block_k != 128)
        return fail(err, GEMM_ERR_UNSUPPORTED, "block_k must be 0, 64 or 128");
    if (o.group_m < 0 || o.max_clusters < 0 || o.stages < 0)
        return fail(err, GEMM_ERR_INVALID_ARG, "group_m, max_clusters and stages must be >= 0");
    if (o.host_parts < 0 || o.host_parts > kHostChunks)
        return fail(err, GEMM_ERR_INVALID_ARG, "host_parts must be between 0 and %d", kHostChunks);
    if (o.clock_probe != 0 && o.clock_probe != 1)
        return fail(err, GEMM_ERR_INVALID_ARG, "clock_probe must be 0 or 1");
    if (o.schedule < 0 || o.schedule > 3)
        return fail(err, GEMM_ERR_INVALID_ARG,
                    "schedule must be 0 (auto), 1 (whole tiles), 2 (stream-K tail) or 3 (cluster launch control)");
    if (M < 0 || N < 0 || K < 0 || batch < 0)
        return fail(err, GEMM_ERR_INVALID_ARG, "negative size");
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31) || batch >= (1ll << 31))
        return fail(err, GEMM_ERR_INVALID_ARG, "every dimension must be below 2^31");

    const bool swap = o.layout_c == GEMM_COL_MAJOR;
    const int cm = swap ? o.cluster_n : o.cluster_m;
    const int cn = swap ? o.cluster_m : o.cluster_n;
    // Auto: the pair MMA wherever the cluster's M extent is even. Each CTA then feeds
    // its tensor core half of B's columns per k-step, which unloads the shared-memory
    // port that bounds single-CTA tiles (4096^3 in 2x1 clusters: 1764 against 1556
    // TFLOP/s with B multicast instead).
    const int G = o.cta_group ? o.cta_group : ((cm & 1) ? 1 : 2);
    if (G == 2 && (cm & 1))
        return fail(err, GEMM_ERR_UNSUPPORTED,
                    "cta_group 2 pairs CTAs along M: the cluster extent along M%s must be even",
                    swap ? " (cluster_n, since column-major C swaps M and N)" : "");
    int ma = o.mode == GEMM_MODE_MCAST ? (swap ? o.mcast_b : o.mcast_a) : 0;
    int mb = o.mode == GEMM_MODE_MCAST ? (swap ? o.mcast_a : o.mcast_b) : 0;
    const int gA = ma ? cn : 1;
    const int gB = mb ? cm / G : 1;
    if (gA == 1) ma = 0;
    if (gB == 1) mb = 0;

    const int BN = o.block_n ? o.block_n : 256;
    // 1024 for aligning the dynamic base, the epilogue staging, then per stage a
    // full and an empty barrier, plus 9 barriers (accumulators, drain, and one per
    // epilogue warp for staging stream-K partials), the TMEM address, the abort
    // flag and the epilogue warps' agreement words.
    const int fixed = 1024 + dgc::EPI_SMEM_BYTES + 9 * 8 + 32 + 256;   // + the tile-id ring
    auto stage_bytes_for = [&](int bk) { return dgc::BLOCK_M * bk * 2 + (BN / G) * bk * 2; };
    // Operands as launched (after the C^T transpose): K-major ones need K % 64 == 0
    // for the k-split map that 128-wide stages use.
    const bool a_kmajor = (swap ? o.layout_b == GEMM_COL_MAJOR : o.layout_a == GEMM_ROW_MAJOR);
    const bool b_kmajor = (swap ? o.layout_a == GEMM_ROW_MAJOR : o.layout_b == GEMM_COL_MAJOR);
    const bool k_split_ok = (K % dgc::ATOM_K) == 0 || (!a_kmajor && !b_kmajor);
    int BK = o.block_k;
    if (BK == 0) {
        // 128-wide stages halve the producers' per-byte issue cost; keep them when
        // at least three still fit in shared memory.
        BK = (k_split_ok && (kMaxSmemPerCta - fixed) / (stage_bytes_for(128) + 16) >= 3) ? 128 : 64;
    }
    if (BK == 128 && !k_split_ok)
        return fail(err, GEMM_ERR_UNSUPPORTED, "block_k 128 needs K a multiple of 64 when an operand is K-major");
    const int stage_bytes = stage_bytes_for(BK);
    int S = o.stages;
    const int max_s = (kMaxSmemPerCta - fixed) / (stage_bytes + 16);
    if (S == 0) S = max_s < 8 ? max_s : 8;
    if (S < 2 || S > max_s || S > 16)
        return fail(err, GEMM_ERR_UNSUPPORTED, "stages %d: between 2 and %d fit in shared memory", S, max_s);

    r.M = swap ? N : M;
    r.N = swap ? M : N;
    r.K = K;
    r.mcast_a = ma;
    r.mcast_b = mb;
    // A' = B^T when swapped: B row-major (N contiguous) becomes an M'-contiguous A'.
    const int la = swap ? (o.layout_b == GEMM_ROW_MAJOR ? GEMM_COL_MAJOR : GEMM_ROW_MAJOR) : o.layout_a;
    const int lb = swap ? (o.layout_a == GEMM_ROW_MAJOR ? GEMM_COL_MAJOR : GEMM_ROW_MAJOR) : o.layout_b;
    r.a_mn = la == GEMM_COL_MAJOR;   // A' (M' x K) column-major: M' contiguous
    r.b_mn = lb == GEMM_ROW_MAJOR;   // B' (K x N') row-major: N' contiguous
    r.out_f32 = o.out_type == GEMM_OUT_F32;

    gemm_plan_t& p = r.pub;
    memset(&p, 0, sizeof p);
    p.block_m = dgc::BLOCK_M;
    p.block_n = BN;
    p.block_k = BK;
    p.stages = S;
    p.smem_bytes = fixed + S * (stage_bytes + 16);
    p.cluster_m = cm;
    p.cluster_n = cn;
    p.cta_group = G;
    p.group_a = gA;
    p.group_b = gB;
    p.transposed = swap ? 1 : 0;
    const int64_t tm = ceil_div(r.M, (int64_t)cm * dgc::BLOCK_M);
    const int64_t tn = ceil_div(r.N, (int64_t)cn * BN);
    p.tiles = tm * tn * batch;
    int64_t clusters = sm_count / (cm * cn);
    if (o.max_clusters > 0 && o.max_clusters < clusters) clusters = o.max_clusters;
    if (p.tiles < clusters) {
        // Fewer tiles than clusters. Whole tiles leave the rest idle. The stream-K
        // schedule spreads the k-blocks over more clusters, at least kMinSplitBlocks
        // each so small problems stay compact; auto does so only when at most half
        // the clusters would have a tile. (Handing a partial to the finisher costs
        // a few microseconds at the end of the kernel.)
        const int64_t num_kb = ceil_div(K, (int64_t)BK);
        int64_t want = p.tiles;
        if (num_kb >= 2 && (o.schedule == 2 || (o.schedule == 0 && 2 * p.tiles <= clusters))) {
            const int64_t spread = p.tiles * num_kb / kMinSplitBlocks;
            if (spread > want) want = spread;
        }
        if (want < clusters) clusters = want;
    }
    p.clusters = clusters;
    const int64_t k_pad = ceil_div(K, BK) * BK;
    p.l2_to_sm_operand_bytes = p.tiles * cm * cn * k_pad * 2 * (dgc::BLOCK_M / gA + (BN / G) / gB);
    p.stream_k_tiles = 0;
    // L2 eviction priorities. When every cluster tile has the same column block (one
    // tile along N), each A row block is read by one tile only: A streams through L2
    // once (evict first) while B, which every tile reads, stays (evict last); the
    // mirror case for one tile along M. Measured on the skinny GEMMs (16384 x 128 x
    // 8192 and 128 x 16384 x 8192): 52 -> 49-50 us. Elsewhere no hint: on 8192^3 the
    // hinted loads ran 5% slower and read as many DRAM bytes.
    p.l2_hint_a = p.l2_hint_b = dgc::L2_HINT_NONE;
    p.k_rotate = 0;
    if (batch == 1 && tm > 1 && tn == 1) {
        p.l2_hint_a = dgc::L2_HINT_EVICT_FIRST;
        p.l2_hint_b = dgc::L2_HINT_EVICT_LAST;
        // K-major A rows of different tiles share no DRAM pages; start each tile at its
        // own k-block so the tiles do not all ask L2 for the same B k-block at once. (A
        // rotated tile sums its k-blocks in another order, so it rounds differently from
        // a launch whose tile grid is not one tile wide.)
        p.k_rotate = r.a_mn ? 0 : 1;
    } else if (batch == 1 && tm == 1 && tn > 1) {
        // No rotation here: an MN-major B is read in lockstep by neighbouring tiles, whose
        // rows share DRAM pages (measured on 128 x 16384 x 8192: rotation cost 2 us).
        p.l2_hint_a = dgc::L2_HINT_EVICT_LAST;
        p.l2_hint_b = dgc::L2_HINT_EVICT_FIRST;
    }
    // Serpentine k walk: in the raster band a cluster's next whole tile reuses its A
    // rows a wave later, after the whole K range of a wave's operands has passed
    // through L2. Walking k backwards on every other tile starts it on the k-blocks
    // read last. Only for long K (at least 16 k-blocks) and at least two waves of
    // whole tiles, where those re-reads come from DRAM (8192^3 pair + 4-CTA
    // multicast: DRAM 1.41 -> 1.25 GB per launch, 588 -> 582 us; 4096^3 pair 79.1 -> 77.9 us;
    // neither slower anywhere measured). The bands snake as well (odd bands walk their
    // columns from the last, starting on the B columns L2 received last: 1.25 -> 1.17 GB,
    // 598 -> 594 us on 8192^3). A reversed tile sums
    // its k-blocks in the other order, so it rounds differently from the same tile of
    // a launch that walks it forwards.
    p.k_serpentine = (p.l2_hint_a == dgc::L2_HINT_NONE && ceil_div(K, BK) >= 16 && clusters > 0 &&
                      p.tiles >= 2 * clusters) ? 1 : 0;
    // Each producer prefetches the first k-blocks of its first tile into L2 before
    // waiting for the previous grid: back to back, a launch's first DRAM reads overlap
    // its predecessor's last tiles. A ring's worth in general (16384 x 128 x 8192:
    // 48.5 -> 47.2 us; 4096^3: 90.3 -> 89.2 us; deeper was 0.5 % slower there; 8192^3
    // and the attention-score batch unchanged); three rings' worth where the grid is one
    // tile wide and each tile streams its own operand (16384 x 128 x 8192: 48.1 -> 46.8
    // us, 128 x 16384 x 8192: 46.4 -> 45.9 us; four rings and more crowd L2 and slow both).
    // None with cluster launch control, which launches without programmatic dependent
    // launch.
    p.prefetch_kb = o.schedule == 3 ? 0 : (p.l2_hint_a != dgc::L2_HINT_NONE ? 3 : 1) * S;
    return GEMM_OK;
}

// Whole-tile waves and the stream-K tail for `tiles` cluster tiles on `clusters`
// co-resident clusters of `cs` CTAs. Returns the number of tiles processed whole
// (a multiple of `clusters`); the rest are split by k-blocks. The auto schedule
// splits when that saves at least kMinTailUs: whole tiles take `waves` cluster-
// tile times, an even split tiles / clusters of them, a cluster tile's time being
// its FLOPs at cs SMs' share of the tensor rate. (Handing a partial to its
// finisher costs a few microseconds, so a short tail is cheaper left idle.)
int64_t whole_tiles_for(int schedule, int64_t tiles, int64_t clusters, int num_kb, bool can_split, double flops,
                        int cs) {
    if (!can_split || schedule == 1 || schedule == 3 || num_kb < 2 || tiles == 0 || clusters <= 1) return tiles;
    const int64_t waves = (tiles + clusters - 1) / clusters;
    const double tile_us = flops / (double)tiles / (kFlopPerUsPerSm * cs);
    const double saved_us = ((double)waves - (double)tiles / (double)clusters) * tile_us;
    if (schedule == 0 && saved_us < kMinTailUs) return tiles;
    const int64_t full = tiles / clusters;
    return (full > 0 ? full - 1 : 0) * clusters;
}

template <int BN, int G, int BK>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&dgc::dgc_gemm_kernel<BN, G, BK>);
}

template <int BK>
void* pick_kernel_bk(int BN, int G) {
    if (BN == 256) return G == 1 ? kernel_ptr<256, 1, BK>() : kernel_ptr<256, 2, BK>();
    return G == 1 ? kernel_ptr<128, 1, BK>() : kernel_ptr<128, 2, BK>();
}

void* pick_kernel(int BN, int G, int BK) {
    return BK == 128 ? pick_kernel_bk<128>(BN, G) : pick_kernel_bk<64>(BN, G);
}

// K == 0: C <- beta * C (zero when beta == 0, without reading C).
__global__ void scale_c_kernel(void* C, int64_t rows, int64_t cols, int64_t ldc, int64_t stride,
                               int64_t batch, int f32, float beta) {
    const int64_t per = rows * cols;
    const int64_t total = per * batch;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / per, rc = i - b * per, r = rc / cols, c = rc - r * cols;
        const int64_t off = b * stride + r * ldc + c;
        if (f32) {
            float* p = static_cast<float*>(C) + off;
            *p = beta == 0.0f ? 0.0f : beta * *p;
        } else {
            uint16_t* p = static_cast<uint16_t*>(C) + off;
            float v = beta == 0.0f ? 0.0f : beta * __uint_as_float((uint32_t)*p << 16);
            *p = (uint16_t)(dgc::pack_bf16x2(v, 0.0f) & 0xFFFFu);
        }
    }
}

}  // namespace

static const char* kStatusNames[] = {
    "GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_UNSUPPORTED", "GEMM_ERR_ALIGNMENT",
    "GEMM_ERR_CUDA", "GEMM_ERR_DEVICE_TIMEOUT", "GEMM_ERR_NOT_SM103"};

extern "C" const char* gemm_status_string(gemm_status_t s) {
    if ((int)s < 0 || (int)s >= (int)(sizeof kStatusNames / sizeof kStatusNames[0])) return "GEMM_ERR_UNKNOWN";
    return kStatusNames[s];
}

extern "C" const char* gemm_last_error(gemm_handle_t h) {
    return h ? h->err.c_str() : g_thread_error.c_str();
}

extern "C" void gemm_options_default(gemm_options_t* o) {
    if (!o) return;
    memset(o, 0, sizeof *o);
    o->mode = GEMM_MODE_UNICAST;
    o->cluster_m = 1;
    o->cluster_n = 1;
    o->cta_group = 1;
    o->layout_a = GEMM_ROW_MAJOR;
    o->layout_b = GEMM_COL_MAJOR;
    o->layout_c = GEMM_ROW_MAJOR;
    o->out_type = GEMM_OUT_BF16;
}

extern "C" gemm_status_t gemm_plan(const gemm_options_t* opt, int64_t M, int64_t N, int64_t K,
                                   int64_t batch, int sm_count, gemm_plan_t* plan) {
    if (!opt || !plan || sm_count <= 0)
        return fail(nullptr, GEMM_ERR_INVALID_ARG, "gemm_plan needs options, a plan and sm_count > 0");
    Resolved r;
    gemm_status_t s = resolve(*opt, M, N, K, batch, sm_count, r, nullptr);
    if (s == GEMM_OK) {
        *plan = r.pub;
        const int num_kb = (int)ceil_div(K, r.pub.block_k);
        plan->stream_k_tiles = r.pub.tiles - whole_tiles_for(opt->schedule, r.pub.tiles, r.pub.clusters, num_kb, true,
                                                             2.0 * (double)M * (double)N * (double)K * (double)batch,
                                                             r.pub.cluster_m * r.pub.cluster_n);
    }
    return s;
}

extern "C" gemm_status_t gemm_create(gemm_handle_t* out, const gemm_options_t* opt, int device) {
    if (!out || !opt) return fail(nullptr, GEMM_ERR_INVALID_ARG, "gemm_create needs out and opt");
    *out = nullptr;
    Resolved r;
    gemm_status_t s = resolve(*opt, 0, 0, 0, 1, 1, r, nullptr);
    if (s != GEMM_OK) return s;
    if (opt->mode == GEMM_MODE_MCAST && (opt->mcast_a || opt->mcast_b) && world_is_multi_gpu())
        return fail(nullptr, GEMM_ERR_UNSUPPORTED,
                    "cluster multicast is single-GPU only; WORLD_SIZE > 1 requires unicast or the pair MMA");
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess)
        return fail(nullptr, GEMM_ERR_CUDA, "cudaGetDeviceProperties(%d): %s", device, cudaGetErrorString(e));
    if (prop.major != 10 || prop.minor != 3)
        return fail(nullptr, GEMM_ERR_NOT_SM103, "device %d is sm_%d%d; this library is built for sm_103a",
                    device, prop.major, prop.minor);
    gemm_handle_s* h = new gemm_handle_s();
    h->opt = *opt;
    if (h->opt.wait_timeout_ns == 0) h->opt.wait_timeout_ns = kDefaultTimeoutNs;
    h->device = device;
    h->sm_count = prop.multiProcessorCount;
    memset(h->occ_key, 0, sizeof h->occ_key);
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(device);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        cudaSetDevice(prev);
        delete h;
        return fail(nullptr, GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    e = cudaMalloc(&h->d_status, 16);
    if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, 16);
    if (e == cudaSuccess && opt->clock_probe) {
        e = cudaMalloc(&h->d_clock, kClockBytes);
        if (e == cudaSuccess) e = cudaMemset(h->d_clock, 0, kClockBytes);
    }
    if (e != cudaSuccess) {
        if (h->d_status) cudaFree(h->d_status);   // with the handle's device current
        if (h->d_clock) cudaFree(h->d_clock);
        cudaSetDevice(prev);
        delete h;
        return fail(nullptr, GEMM_ERR_CUDA, "status word / clock counters: %s", cudaGetErrorString(e));
    }
    cudaSetDevice(prev);
    *out = h;
    return GEMM_OK;
}

extern "C" gemm_status_t gemm_destroy(gemm_handle_t h) {
    if (!h) return GEMM_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    if (h->d_status) cudaFree(h->d_status);
    if (h->d_clock) cudaFree(h->d_clock);
    if (h->workspace) cudaFree(h->workspace);
    if (h->flags) cudaFree(h->flags);
    for (int i = 0; i < 3; ++i)
        if (h->stage_ptr[i]) cudaFree(h->stage_ptr[i]);
    if (h->pipe_ready) {
        cudaStreamDestroy(h->pipe_in);
        cudaStreamDestroy(h->pipe_out);
        cudaEventDestroy(h->ev_start);
        cudaEventDestroy(h->ev_whole);
        cudaEventDestroy(h->ev_out_done);
        for (int i = 0; i < kHostChunks; ++i) {
            cudaEventDestroy(h->ev_in[i]);
            cudaEventDestroy(h->ev_c[i]);
        }
    }
    cudaSetDevice(prev);
    delete h;
    return GEMM_OK;
}

extern "C" int64_t gemm_launch_count(gemm_handle_t h) { return h ? h->launches : -1; }

extern "C" int64_t gemm_schedule_work(int64_t tiles, int64_t dp_tiles, int num_kb, int64_t clusters,
                                      int64_t cluster, gemm_work_item_t* items, int64_t capacity) {
    if (tiles < 0 || dp_tiles < 0 || dp_tiles > tiles || num_kb < 1 || clusters < 1 || cluster < 0 ||
        cluster >= clusters || capacity < 0 || (capacity > 0 && !items))
        return -1;
    // The same iterator the kernel's roles walk, replayed on the host.
    dgc::KernelParams kp;
    memset(&kp, 0, sizeof kp);
    kp.num_kb = num_kb;
    kp.total_tiles = tiles;
    kp.dp_tiles = dp_tiles;
    kp.sk_iters = (tiles - dp_tiles) * (int64_t)num_kb;
    dgc::WorkIter wi;
    wi.init(kp, cluster, clusters, nullptr);
    dgc::Work w;
    int64_t n = 0;
    while (wi.next(kp, w)) {
        if (n < capacity) {
            gemm_work_item_t& it = items[n];
            it.tile = w.tile;
            it.kb0 = w.kb0;
            it.kb1 = w.kb1;
            it.kind = w.kind;
            it.contrib_first = w.kind == dgc::WORK_FINISHER ? w.contrib_first : -1;
            it.contrib_count = w.kind == dgc::WORK_FINISHER ? w.contrib_count : 0;
            it.last = w.last ? 1 : 0;
        }
        ++n;
    }
    return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Encodes a 3-D tiled map (inner, outer, batch) with the 128-byte swizzle.
static gemm_status_t encode_map(gemm_handle_s* h, CUtensorMap* map, CUtensorMapDataType dt, int esize,
                                const void* ptr, int64_t inner, int64_t outer, int64_t batch,
                                int64_t ld, int64_t stride, uint32_t box_inner, uint32_t box_outer,
                                const char* what) {
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
    int64_t bstride = batch > 1 ? stride : ((ld * outer + 15) / 16) * 16;
    if (bstride <= 0) bstride = 16;
    cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(bstride * esize)};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = h->encode(map, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(&h->err, GEMM_ERR_INVALID_ARG,
                    "cuTensorMapEncodeTiled(%s) failed with %d (dims %lld x %lld x %lld, ld %lld, stride %lld)",
                    what, (int)res, (long long)inner, (long long)outer, (long long)batch, (long long)ld,
                    (long long)stride);
    return GEMM_OK;
}

// Encodes the k-split view of a K-major bf16 operand (K a multiple of 64):
// dims {64 K, rows, K/64, batch} with the 64-element atoms 128 bytes apart, so one
// box {64, box_rows, box_atoms, 1} lands as box_atoms consecutive swizzled tiles.
static gemm_status_t encode_ksplit(gemm_handle_s* h, CUtensorMap* map, const void* ptr, int64_t K, int64_t rows,
                                   int64_t batch, int64_t ld, int64_t stride, uint32_t box_rows, uint32_t box_atoms,
                                   const char* what) {
    cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64), (cuuint64_t)batch};
    int64_t bstride = batch > 1 ? stride : ((ld * rows + 15) / 16) * 16;
    if (bstride <= 0) bstride = 16;
    cuuint64_t strides[3] = {(cuuint64_t)(ld * 2), 128, (cuuint64_t)(bstride * 2)};
    cuuint32_t box[4] = {64, box_rows, box_atoms, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult res = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS)
        return fail(&h->err, GEMM_ERR_INVALID_ARG,
                    "cuTensorMapEncodeTiled(%s, k-split) failed with %d (K %lld, rows %lld, batch %lld, ld %lld)",
                    what, (int)res, (long long)K, (long long)rows, (long long)batch, (long long)ld);
    return GEMM_OK;
}

// Box of one issuer's slice of a K-major tile of `rows` rows and `atoms` atoms
// shared by `parts` issuers: whole atoms first, then bands of rows.
static void ksplit_box(int rows, int atoms, int parts, uint32_t& box_rows, uint32_t& box_atoms) {
    if (parts <= atoms) {
        box_rows = (uint32_t)rows;
        box_atoms = (uint32_t)(atoms / parts);
    } else {
        box_rows = (uint32_t)(rows / (parts / atoms));
        box_atoms = 1;
    }
}

gemm_status_t dgc_host::run_impl(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                 int64_t strideA, const void* B, int64_t ldb, int64_t strideB, void* C,
                                 int64_t ldc, int64_t strideC, int64_t batch, float alpha, float beta,
                                 void* stream_v) {
    if (!h) return fail(nullptr, GEMM_ERR_INVALID_ARG, "null handle");
    const gemm_options_t& o = h->opt;
    Resolved r;
    gemm_status_t s = resolve(o, M, N, K, batch, h->sm_count, r, &h->err);
    if (s != GEMM_OK) return s;
    if (M == 0 || N == 0 || batch == 0) return GEMM_OK;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    const int esc = o.out_type == GEMM_OUT_F32 ? 4 : 2;

    // ---- argument checks (user's view: A M x K, B K x N, C M x N)
    if (!C) return fail(&h->err, GEMM_ERR_INVALID_ARG, "C is null");
    if (K > 0 && (!A || !B)) return fail(&h->err, GEMM_ERR_INVALID_ARG, "A or B is null");
    const int64_t a_inner = o.layout_a == GEMM_ROW_MAJOR ? K : M;
    const int64_t a_outer = o.layout_a == GEMM_ROW_MAJOR ? M : K;
    const int64_t b_inner = o.layout_b == GEMM_ROW_MAJOR ? N : K;
    const int64_t b_outer = o.layout_b == GEMM_ROW_MAJOR ? K : N;
    const int64_t c_inner = o.layout_c == GEMM_ROW_MAJOR ? N : M;
    const int64_t c_outer = o.layout_c == GEMM_ROW_MAJOR ? M : N;
    if (ldc < c_inner || ldc < 1) return fail(&h->err, GEMM_ERR_INVALID_ARG, "ldc %lld < %lld", (long long)ldc, (long long)c_inner);
    if (!aligned16(C) || (ldc * esc) % 16)
        return fail(&h->err, GEMM_ERR_ALIGNMENT, "C must be 16-byte aligned with ldc*%d a multiple of 16", esc);
    if (batch > 1) {
        if ((strideC * esc) % 16 || strideC < ldc * c_outer)
            return fail(&h->err, strideC < ldc * c_outer ? GEMM_ERR_INVALID_ARG : GEMM_ERR_ALIGNMENT,
                        "strideC must be a multiple of 16 bytes and keep batches of C apart");
    }
    if (K > 0) {
        if (lda < a_inner || lda < 1) return fail(&h->err, GEMM_ERR_INVALID_ARG, "lda %lld < %lld", (long long)lda, (long long)a_inner);
        if (ldb < b_inner || ldb < 1) return fail(&h->err, GEMM_ERR_INVALID_ARG, "ldb %lld < %lld", (long long)ldb, (long long)b_inner);
        if (!aligned16(A) || !aligned16(B) || (lda * 2) % 16 || (ldb * 2) % 16)
            return fail(&h->err, GEMM_ERR_ALIGNMENT,
                        "A and B must be 16-byte aligned with lda*2 and ldb*2 multiples of 16");
        if (batch > 1 && ((strideA * 2) % 16 || (strideB * 2) % 16 || strideA < 0 || strideB < 0))
            return fail(&h->err, GEMM_ERR_ALIGNMENT, "strideA*2 and strideB*2 must be non-negative multiples of 16");
        // A stride of 0 shares one matrix across the batch; any other stride must keep the
        // matrices apart (a tensor map cannot describe overlapping ones).
        if (batch > 1 && ((strideA != 0 && strideA < lda * a_outer) || (strideB != 0 && strideB < ldb * b_outer)))
            return fail(&h->err, GEMM_ERR_INVALID_ARG,
                        "strideA and strideB must be 0 (one matrix for every product) or keep the matrices apart");
    }

    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    struct Restore {
        int d, p;
        ~Restore() { if (d != p) cudaSetDevice(p); }
    } restore{h->device, prev};

    if (K == 0) {
        const int64_t total = M * N * batch;
        const int threads = 256;
        const int64_t blocks = total / threads + 1 < 4096 ? total / threads + 1 : 4096;
        // Row-major view of C: rows x cols with leading dimension ldc.
        scale_c_kernel<<<(unsigned)blocks, threads, 0, stream>>>(C, c_outer, c_inner, ldc, strideC, batch,
                                                                 o.out_type == GEMM_OUT_F32, beta);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "scale launch: %s", cudaGetErrorString(e));
        h->launches++;
        return GEMM_OK;
    }

    // ---- operands as launched (column-major C computes C^T = B^T A^T)
    Operand opA{A, lda, strideA, o.layout_a == GEMM_COL_MAJOR};
    Operand opB{B, ldb, strideB, o.layout_b == GEMM_ROW_MAJOR};
    if (r.pub.transposed) {
        // A' = B^T (N x K): B row-major has N contiguous -> M'-major.
        // B' = A^T (K x M): A row-major has K contiguous -> K-major.
        Operand a2{B, ldb, strideB, o.layout_b == GEMM_ROW_MAJOR};
        Operand b2{A, lda, strideA, o.layout_a == GEMM_COL_MAJOR};
        opA = a2;
        opB = b2;
    }
    const gemm_plan_t& pl = r.pub;
    const int BN = pl.block_n, G = pl.cta_group;
    const int gA = pl.group_a, gB = pl.group_b;

    const int BK = pl.block_k;
    const int atoms = BK / dgc::ATOM_K;
    const bool kmap4 = (r.K % dgc::ATOM_K) == 0;
    // An operand shared by every product is mapped as a single matrix.
    const bool a_shared = batch > 1 && opA.stride == 0, b_shared = batch > 1 && opB.stride == 0;
    const int64_t batch_a = a_shared ? 1 : batch, batch_b = b_shared ? 1 : batch;
    CUtensorMap tmA, tmB, tmC;
    uint32_t br, ba;
    if (!opA.mn_major && kmap4) {
        ksplit_box(dgc::BLOCK_M, atoms, gA, br, ba);
        s = encode_ksplit(h, &tmA, opA.ptr, r.K, r.M, batch_a, opA.ld, opA.stride, br, ba, "A");
    } else if (!opA.mn_major) {
        s = encode_map(h, &tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, opA.ptr, r.K, r.M, batch_a, opA.ld, opA.stride,
                       64, dgc::BLOCK_M / gA, "A");
    } else {
        s = encode_map(h, &tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, opA.ptr, r.M, r.K, batch_a, opA.ld, opA.stride,
                       64, BK / gA, "A");
    }
    if (s != GEMM_OK) return s;
    if (!opB.mn_major && kmap4) {
        ksplit_box(BN / G, atoms, gB, br, ba);
        s = encode_ksplit(h, &tmB, opB.ptr, r.K, r.N, batch_b, opB.ld, opB.stride, br, ba, "B");
    } else if (!opB.mn_major) {
        s = encode_map(h, &tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, opB.ptr, r.K, r.N, batch_b, opB.ld, opB.stride,
                       64, (BN / G) / gB, "B");
    } else {
        s = encode_map(h, &tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, opB.ptr, r.N, r.K, batch_b, opB.ld, opB.stride,
                       64, BK / gB, "B");
    }
    if (s != GEMM_OK) return s;
    s = encode_map(h, &tmC, r.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, esc,
                   C, r.N, r.M, batch, ldc, strideC, r.out_f32 ? 32 : 64, 32, "C");
    if (s != GEMM_OK) return s;

    dgc::KernelParams kp;
    memset(&kp, 0, sizeof kp);
    kp.M = (int)r.M;
    kp.N = (int)r.N;
    kp.K = (int)r.K;
    kp.batch = (int)batch;
    kp.num_kb = (int)ceil_div(r.K, BK);
    kp.a_kmap4 = !opA.mn_major && kmap4;
    kp.b_kmap4 = !opB.mn_major && kmap4;
    kp.a_shared = a_shared ? 1 : 0;
    kp.b_shared = b_shared ? 1 : 0;
    kp.cx = pl.cluster_m;
    kp.cy = pl.cluster_n;
    kp.mcast_a = r.mcast_a;
    kp.mcast_b = r.mcast_b;
    kp.a_mn_major = opA.mn_major;
    kp.b_mn_major = opB.mn_major;
    kp.out_f32 = r.out_f32;
    kp.tiles_m = (int)ceil_div(r.M, (int64_t)pl.cluster_m * dgc::BLOCK_M);
    kp.tiles_n = (int)ceil_div(r.N, (int64_t)pl.cluster_n * BN);
    kp.total_tiles = pl.tiles;
    kp.group_m = o.group_m > 0 ? o.group_m : 4;   // measured best on 4096^3 and 8192^3 (fewest DRAM re-reads)
    kp.stages = pl.stages;
    kp.debug_flags = o.debug_flags;
    kp.alpha = alpha;
    kp.beta = beta;
    kp.c_in = C;
    kp.ldc = ldc;
    kp.stride_c = strideC;
    kp.status = h->d_status;
    kp.timeout_ns = o.wait_timeout_ns;
    kp.a_l2 = pl.l2_hint_a;
    kp.b_l2 = pl.l2_hint_b;
    kp.k_rotate = pl.k_rotate;
    kp.k_serpentine = pl.k_serpentine;
    kp.prefetch_kb = pl.prefetch_kb;
    kp.clk = h->d_clock;

    void* fn = pick_kernel(BN, G, BK);
    const int bi = BN == 256 ? 1 : 0, gi = G - 1, ki = BK == 128 ? 1 : 0;
    if (!h->smem_set[bi][gi][ki]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemPerCta);
        if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
        h->smem_set[bi][gi][ki] = true;
    }
    const int cs = pl.cluster_m * pl.cluster_n;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: this grid may be scheduled while the previous
    // kernel in the stream finishes; the kernel waits for that kernel's completion
    // (griddepcontrol.wait) before its first global memory access. Not with cluster
    // launch control, whose pending clusters must not compete with a next grid.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(dgc::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int& occ = h->occ_key[bi][gi][ki][cs];
    if (occ == 0) {
        cfg.gridDim = dim3((unsigned)(cs * (h->sm_count / cs)), 1, 1);
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess || n <= 0)
            return fail(&h->err, GEMM_ERR_CUDA, "cudaOccupancyMaxActiveClusters: %s (n=%d)",
                        cudaGetErrorString(e), n);
        occ = n;
    }
    int64_t clusters = pl.clusters < occ ? pl.clusters : occ;
    if (o.schedule == 3) {
        // One cluster per tile; the resident ones take the pending ones' tiles.
        clusters = pl.tiles;
        kp.clc = 1;
    }
    // Stream-K tail (needs the co-residency the occupancy cap guarantees, and a workspace).
    if (o.schedule == 2 && h->no_alloc)
        return fail(&h->err, GEMM_ERR_UNSUPPORTED, "the stream-K tail needs a workspace; gemm_run_noalloc runs whole tiles");
    kp.dp_tiles = whole_tiles_for(o.schedule, pl.tiles, clusters, kp.num_kb, !h->no_alloc,
                                  2.0 * (double)M * (double)N * (double)K * (double)batch, cs);
    kp.sk_iters = (pl.tiles - kp.dp_tiles) * kp.num_kb;
    if (kp.sk_iters == 0 && o.schedule != 3 && clusters > pl.tiles) clusters = pl.tiles;   // whole tiles only
    cfg.gridDim = dim3((unsigned)(clusters * cs), 1, 1);
    if (kp.sk_iters > 0) {
        const size_t slots = (size_t)(clusters * cs);
        const size_t ws_bytes = slots * dgc::BLOCK_M * BN * sizeof(float);
        if (ws_bytes > h->workspace_bytes) {
            if (h->workspace) cudaFree(h->workspace);
            h->workspace = nullptr;
            h->workspace_bytes = 0;
            cudaError_t e = cudaMalloc(&h->workspace, ws_bytes);
            if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "stream-K workspace: %s", cudaGetErrorString(e));
            h->workspace_bytes = ws_bytes;
        }
        if (slots > h->flag_count) {
            if (h->flags) cudaFree(h->flags);
            h->flags = nullptr;
            h->flag_count = 0;
            cudaError_t e = cudaMalloc(&h->flags, slots * sizeof(unsigned int));
            if (e == cudaSuccess) e = cudaMemset(h->flags, 0, slots * sizeof(unsigned int));
            if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "stream-K flags: %s", cudaGetErrorString(e));
            h->flag_count = slots;
        }
        kp.workspace = h->workspace;
        kp.flags = h->flags;
    }
    cfg.numAttrs = o.schedule == 3 ? 1 : 2;
    if (h->no_alloc) {
        // The shared static record must start at zero; cleared only now, when every
        // check has passed and a launch follows, so a refused call writes nothing.
        cudaError_t e = cudaMemsetAsync(h->d_status, 0, 16, stream);
        if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "clearing the status record: %s", cudaGetErrorString(e));
        h->status_cleared = true;
    }
    void* args[] = {&tmA, &tmB, &tmC, &kp};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "cudaLaunchKernelEx: %s", cudaGetErrorString(e));
    h->launches++;
    return GEMM_OK;
}

extern "C" gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                  const void* B, int64_t ldb, void* C, int64_t ldc, float alpha, float beta,
                                  void* stream) {
    return run_impl(h, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, alpha, beta, stream);
}

extern "C" gemm_status_t gemm_run_strided_batched(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                                  const void* A, int64_t lda, int64_t strideA, const void* B,
                                                  int64_t ldb, int64_t strideB, void* C, int64_t ldc,
                                                  int64_t strideC, int64_t batch, float alpha, float beta,
                                                  void* stream) {
    return run_impl(h, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch, alpha, beta, stream);
}

extern "C" gemm_status_t gemm_query_status(gemm_handle_t h, void* stream_v) {
    if (!h) return fail(nullptr, GEMM_ERR_INVALID_ARG, "null handle");
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    struct Restore {
        int d, p;
        ~Restore() { if (d != p) cudaSetDevice(p); }
    } restore{h->device, prev};
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream_v));
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    unsigned int w[4] = {0, 0, 0, 0};
    e = cudaMemcpy(w, h->d_status, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (w[0] == 0) return GEMM_OK;
    static const char* roles[] = {"none", "producer waiting for a free stage", "MMA waiting for stage bytes",
                                  "MMA waiting for a free accumulator", "epilogue waiting for an accumulator",
                                  "teardown waiting for in-flight MMAs",
                                  "stream-K finisher waiting for another cluster's partial",
                                  "a role waiting for a tile id from cluster launch control",
                                  "the scheduler waiting for a free tile-id slot",
                                  "stream-K finisher waiting for partials copied into shared memory"};
    const char* role = w[0] < 10 ? roles[w[0]] : "unknown";
    fail(&h->err, GEMM_ERR_DEVICE_TIMEOUT, "bounded wait expired: %s (stage/buffer %u, CTA %u, tile %d)", role,
         w[1], w[2], (int)w[3]);
    cudaMemset(h->d_status, 0, 16);
    // An aborted launch may leave stream-K flags raised; lower them for the next one.
    if (h->flags) cudaMemset(h->flags, 0, h->flag_count * sizeof(unsigned int));
    return GEMM_ERR_DEVICE_TIMEOUT;
}

extern "C" gemm_status_t gemm_read_clock(gemm_handle_t h, void* stream_v, uint64_t out[3]) {
    if (!h || !out) return fail(h ? &h->err : nullptr, GEMM_ERR_INVALID_ARG, "gemm_read_clock needs a handle and out");
    if (!h->d_clock) return fail(&h->err, GEMM_ERR_INVALID_ARG, "the handle was created without clock_probe");
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != h->device) cudaSetDevice(h->device);
    struct Restore {
        int d, p;
        ~Restore() { if (d != p) cudaSetDevice(p); }
    } restore{h->device, prev};
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream_v));
    unsigned long long c[3 * dgc::CLOCK_PROBE_SLOTS];
    if (e == cudaSuccess) e = cudaMemcpy(c, h->d_clock, kClockBytes, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(h->d_clock, 0, kClockBytes);
    if (e != cudaSuccess) return fail(&h->err, GEMM_ERR_CUDA, "clock counters: %s", cudaGetErrorString(e));
    out[0] = out[1] = out[2] = 0;
    for (int sm = 0; sm < dgc::CLOCK_PROBE_SLOTS; ++sm)
        for (int i = 0; i < 3; ++i) out[i] += c[3 * sm + i];
    return GEMM_OK;
}

// ---------------------------------------------------------------------------
// gemm_run_noalloc: gemm_run without a handle and without any device
// allocation. The kernel's status record (16 bytes) lives in this file-scope
// static array instead of handle-owned memory. In host code the array's name is
// only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress, taken once per device with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[256];

namespace {

constexpr size_t kStatusRecordBytes = 16;
static_assert(kStatusRecordBytes <= sizeof(g_noalloc_scratch), "the static array must hold one status record");
constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    void* scratch = nullptr;         // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    bool smem_set[2][2][2] = {};
    int occ[2][2][2][9] = {};
};

NoAllocDevice g_noalloc_dev[kMaxDevices];
std::mutex g_noalloc_mutex;

// One-time set-up on `device`; the caller holds g_noalloc_mutex.
gemm_status_t noalloc_setup(int device) {
    NoAllocDevice& d = g_noalloc_dev[device];
    if (d.ready) return GEMM_OK;
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess)
        return fail(nullptr, GEMM_ERR_CUDA, "cudaGetDeviceProperties(%d): %s", device, cudaGetErrorString(e));
    if (prop.major != 10 || prop.minor != 3)
        return fail(nullptr, GEMM_ERR_NOT_SM103, "device %d is sm_%d%d; this library is built for sm_103a",
                    device, prop.major, prop.minor);
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != device) cudaSetDevice(device);
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (prev != device) cudaSetDevice(prev);
    if (e != cudaSuccess || !ptr)
        return fail(nullptr, GEMM_ERR_CUDA, "cudaGetSymbolAddress(static status record): %s", cudaGetErrorString(e));
    if (e2 != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(nullptr, GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    d.scratch = ptr;
    d.sm_count = prop.multiProcessorCount;
    d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    d.ready = true;
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const gemm_options_t* opt, int device, int64_t M, int64_t N, int64_t K,
                                          const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
                                          int64_t ldc, float alpha, float beta, void* stream,
                                          uint32_t* status_out) {
    if (!opt) return fail(nullptr, GEMM_ERR_INVALID_ARG, "gemm_run_noalloc needs options");
    if (device < 0 || device >= kMaxDevices) return fail(nullptr, GEMM_ERR_INVALID_ARG, "bad device %d", device);
    // Options and sizes first: an impossible request is refused before the device is touched.
    {
        Resolved r;
        gemm_status_t s = resolve(*opt, M, N, K, 1, 1, r, nullptr);
        if (s != GEMM_OK) return s;
    }
    if (opt->schedule == 2)
        return fail(nullptr, GEMM_ERR_UNSUPPORTED, "the stream-K tail needs a workspace; gemm_run_noalloc runs whole tiles");
    if (opt->clock_probe)
        return fail(nullptr, GEMM_ERR_UNSUPPORTED, "the clock probe's counters belong to a handle; gemm_run_noalloc has none");
    if (opt->mode == GEMM_MODE_MCAST && (opt->mcast_a || opt->mcast_b) && world_is_multi_gpu())
        return fail(nullptr, GEMM_ERR_UNSUPPORTED,
                    "cluster multicast is single-GPU only; WORLD_SIZE > 1 requires unicast or the pair MMA");
    // A handle on the host stack that points at the static record: no device memory is allocated.
    gemm_handle_s local;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        gemm_status_t s = noalloc_setup(device);
        if (s != GEMM_OK) return s;
        const NoAllocDevice& d = g_noalloc_dev[device];
        local.opt = *opt;
        if (local.opt.wait_timeout_ns == 0) local.opt.wait_timeout_ns = kDefaultTimeoutNs;
        local.device = device;
        local.no_alloc = true;
        local.sm_count = d.sm_count;
        local.d_status = static_cast<unsigned int*>(d.scratch);
        local.encode = d.encode;
        memcpy(local.smem_set, d.smem_set, sizeof local.smem_set);
        memcpy(local.occ_key, d.occ, sizeof local.occ_key);
    }
    // run_impl clears the record on `stream` right before the GEMM kernel's launch
    // (and only then: an empty problem or K = 0 launches no GEMM and writes no record).
    gemm_status_t s = run_impl(&local, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, alpha, beta, stream);
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoAllocDevice& d = g_noalloc_dev[device];
        memcpy(d.smem_set, local.smem_set, sizeof d.smem_set);
        memcpy(d.occ, local.occ_key, sizeof d.occ);
    }
    if (s != GEMM_OK) {
        g_thread_error = local.err;
        return s;
    }
    if (status_out) {
        if (!local.status_cleared) {
            // No GEMM kernel ran, so no wait could expire; the record was not touched.
            memset(status_out, 0, kStatusRecordBytes);
            return GEMM_OK;
        }
        int prev = 0;
        cudaGetDevice(&prev);
        if (prev != device) cudaSetDevice(device);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cudaError_t e = cudaMemcpyAsync(status_out, local.d_status, kStatusRecordBytes, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (prev != device) cudaSetDevice(prev);
        if (e != cudaSuccess) return fail(nullptr, GEMM_ERR_CUDA, "reading the status record: %s", cudaGetErrorString(e));
        if (status_out[0] != 0)
            return fail(nullptr, GEMM_ERR_DEVICE_TIMEOUT, "bounded wait expired (code %u, stage/buffer %u, CTA %u)",
                        status_out[0], status_out[1], status_out[2]);
    }
    return GEMM_OK;
}
