// TMA unicast / multicast load microbenchmark for sm_103a (see include/tma_bench.h).
//
// "Hopper TMA Multicast 深度解析与实测", sections 实测 Microbenchmark 源码 and
// 实机运行与 NCU 验证: two scenarios (one tile reloaded, L2-resident; a new
// tile every iteration, DRAM streaming), unicast against multicast. Here every
// CTA keeps `stages` loads in flight (a ring of slots with full/empty
// mbarriers) and one warp consumes: it waits for a slot, checks where the
// 128-byte swizzle put a few elements, and releases the slot to every CTA that
// writes into it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>

#include "densegemm.h"
#include "host_env.h"
#include "ptx.cuh"
#include "tma_bench.h"

namespace {

__device__ unsigned int g_tma_bench_status[4];

struct BenchParams {
    int mode, cluster, box_rows, stages, iters, warmup, stride;
    int tiles_x, tiles_y;
    long long ld;
    const uint16_t* src;
    uint64_t* cycles;
    uint64_t* ns;
    uint32_t* verify;
    uint8_t* landed;             // optional: each CTA's last landed tile, as it sits in shared memory
    int* origin;                 // optional: that tile's (x, y) origin per CTA
    unsigned long long timeout_ns;
};

__device__ bool bench_wait(uint32_t bar, uint32_t parity, const BenchParams& p, uint32_t code) {
    using namespace dgc;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t c0 = clock_cycles();          // budget: 2 SM cycles per ns
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (clock_cycles() - c0 > 2ull * p.timeout_ns) {
            if (atomicCAS(&g_tma_bench_status[0], 0u, code) == 0u) {
                g_tma_bench_status[1] = blockIdx.x;
                __threadfence();
            }
            return false;
        }
    }
}

// Tile of iteration `it`: (it * stride * clusters + cluster id) mod tiles, walked
// incrementally (one conditional subtraction per load instead of a 64-bit
// division, which would cost the issuing thread more than the load itself).
struct TileWalk {
    long long t, step, ntiles;
    __device__ void init(const BenchParams& p, uint32_t cid, uint32_t ncl) {
        ntiles = (long long)p.tiles_x * p.tiles_y;
        t = (long long)cid % ntiles;
        step = ((long long)p.stride * ncl) % ntiles;
    }
    __device__ void next() {
        t += step;
        if (t >= ntiles) t -= ntiles;
    }
    __device__ void origin(const BenchParams& p, int& x, int& y) const {
        x = (int)(t % p.tiles_x) * 64;
        y = (int)(t / p.tiles_x) * p.box_rows;
    }
};

// Release of a slot the consumer did not read: ordering nothing, a relaxed
// arrive avoids the memory barrier a release at cluster scope costs.
__device__ __forceinline__ void arrive_relaxed_cluster(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}

__global__ void __launch_bounds__(64, 1)
tma_bench_kernel(const __grid_constant__ CUtensorMap tm, const BenchParams p) {
    using namespace dgc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    const uint32_t box_bytes = (uint32_t)p.box_rows * 128u;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * box_bytes);
    uint64_t* empty = full + S;
    const uint32_t rank = cluster_ctarank();
    const uint32_t c = (uint32_t)p.cluster;
    const uint32_t cid = cluster_id_x();
    const uint32_t ncl = num_clusters_x();
    const uint16_t all = (uint16_t)((1u << c) - 1u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // unicast: own arm / own consumer; multicast: rank 0 arms, all c consumers
            // release rank 0; sliced: c issuers arm, all c consumers release every issuer.
            mbar_init(smem_u32(&full[s]), p.mode == TMA_BENCH_MULTICAST_SLICED ? c : 1u);
            mbar_init(smem_u32(&empty[s]), p.mode == TMA_BENCH_UNICAST ? 1u : c);
        }
        fence_mbar_init();
    }
    __syncthreads();
    cluster_sync();

    const int total = p.warmup + p.iters;
    bool ok = true;
    if (warp == 0 && lane == 0) {
        const bool issuer = p.mode != TMA_BENCH_MULTICAST || rank == 0;
        if (issuer) {
            prefetch_tmap(&tm);
            const int slice_rows = p.mode == TMA_BENCH_MULTICAST_SLICED ? p.box_rows / (int)c : p.box_rows;
            const uint32_t slice_bytes = (uint32_t)slice_rows * 128u;
            TileWalk tw;
            tw.init(p, cid, ncl);
            int slot = 0;
            uint32_t phase = 0;
            for (int it = 0; ok && it < total; ++it, tw.next()) {
                if (!bench_wait(smem_u32(&empty[slot]), phase ^ 1u, p, 1)) { ok = false; break; }
                int x, y;
                tw.origin(p, x, y);
                const uint32_t fb = smem_u32(&full[slot]);
                const uint32_t dst = smem_u32(smem + slot * box_bytes);
                if (p.mode == TMA_BENCH_UNICAST) {
                    mbar_arrive_expect_tx_local(fb, box_bytes);
                    tma_load_3d(dst, &tm, fb, x, y, 0);
                } else {
                    // Arm every receiver (own barrier and, through mapa, each peer's)
                    // before the one load that feeds them all.
                    for (uint32_t r = 0; r < c; ++r) {
                        if (r == rank) mbar_arrive_expect_tx_local(fb, slice_bytes);
                        else mbar_arrive_expect_tx_cluster(mapa(fb, r), slice_bytes);
                    }
                    if (p.mode == TMA_BENCH_MULTICAST)
                        tma_load_3d_mcast(dst, &tm, fb, x, y, 0, all);
                    else
                        tma_load_3d_mcast(dst + rank * slice_bytes, &tm, fb, x, y + (int)rank * slice_rows, 0, all);
                }
                if (++slot == S) { slot = 0; phase ^= 1u; }
            }
            // Every slot this CTA filled is released by its receivers before exit.
            for (int it = total; ok && it < total + S; ++it) {
                const int slot = it % S;
                if (!bench_wait(smem_u32(&empty[slot]), ((uint32_t)(it / S) & 1u) ^ 1u, p, 1)) break;
            }
        }
    } else if (warp == 1 && lane == 0) {
        uint64_t c0 = 0, g0 = 0;
        uint32_t bad = 0;
        TileWalk tw;
        tw.init(p, cid, ncl);
        int slot = 0;
        uint32_t phase = 0;
        for (int it = 0; it < total; ++it, tw.next()) {
            if (it == p.warmup) {
                c0 = clock64();
                g0 = globaltimer_ns();
            }
            if (!bench_wait(smem_u32(&full[slot]), phase, p, 2)) { ok = false; break; }
            // Every 64th load (and the last), check the first and last row of
            // the tile: element (r, j) of a 128-byte-swizzled box sits at
            // r*128 + ((j/8) ^ (r%8))*16 + (j%8)*2. Checking reads global
            // memory, so it stays off most iterations' critical path.
            const bool check = (it & 63) == 0 || it == total - 1;
            int x = 0, y = 0;
            if (check) tw.origin(p, x, y);
            if (it == total - 1 && p.origin) {
                p.origin[2 * blockIdx.x] = x;
                p.origin[2 * blockIdx.x + 1] = y;
            }
            const uint8_t* box = smem + slot * box_bytes;
            const int rs[2] = {0, p.box_rows - 1};
            const int js[2] = {0, 63};
            for (int a = 0; check && a < 2; ++a) {
                const int r = rs[a], j = js[a];
                const uint16_t got = *reinterpret_cast<const uint16_t*>(
                    box + r * 128 + (((j >> 3) ^ (r & 7)) << 4) + (j & 7) * 2);
                const uint16_t want = p.src[(long long)(y + r) * p.ld + x + j];
                bad += got != want;
            }
            // Release the slot to every CTA that writes into it: a release where this
            // thread read the slot, a relaxed arrive where it did not.
            const uint32_t eb = smem_u32(&empty[slot]);
            if (p.mode == TMA_BENCH_UNICAST) {
                mbar_arrive_local(eb);
            } else if (p.mode == TMA_BENCH_MULTICAST) {
                if (check) mbar_arrive_cluster(mapa(eb, 0));
                else       arrive_relaxed_cluster(mapa(eb, 0));
            } else {
                for (uint32_t r = 0; r < c; ++r) {
                    if (check) mbar_arrive_cluster(mapa(eb, r));
                    else       arrive_relaxed_cluster(mapa(eb, r));
                }
            }
            if (++slot == S) { slot = 0; phase ^= 1u; }
        }
        p.cycles[blockIdx.x] = clock64() - c0;
        p.ns[blockIdx.x] = globaltimer_ns() - g0;
        p.verify[blockIdx.x] = ok ? bad : 0xFFFFFFFFu;
    }
    __syncthreads();
    if (warp == 1 && p.landed && total > 0) {
        // After the timed loop every load has landed and no more are issued: copy the
        // last slot out whole, for a check of every element on the host.
        const int last = (total - 1) % S;
        const uint4* from = reinterpret_cast<const uint4*>(smem + last * box_bytes);
        uint4* to = reinterpret_cast<uint4*>(p.landed + (size_t)blockIdx.x * box_bytes);
        for (uint32_t i = lane; i < box_bytes / 16; i += 32) to[i] = from[i];
    }
    cluster_sync();
}

thread_local char g_err[256];

gemm_status_t bench_fail(gemm_status_t s, const char* msg) {
    snprintf(g_err, sizeof g_err, "%s", msg);
    return s;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

}  // namespace

extern "C" gemm_status_t tma_bench_run(const tma_bench_options_t* opt, const void* src, int64_t rows, int64_t cols,
                                       int64_t ld, uint64_t* cycles, uint64_t* ns, uint32_t* verify,
                                       int* ctas_used, double* delivered_bytes, double* issued_bytes,
                                       void* stream) {
    if (!opt || !src || !cycles || !ns || !verify) return bench_fail(GEMM_ERR_INVALID_ARG, "null argument");
    const tma_bench_options_t& o = *opt;
    int mode = o.mode;
    const int c = o.cluster;
    if (c != 1 && c != 2 && c != 4 && c != 8) return bench_fail(GEMM_ERR_UNSUPPORTED, "cluster must be 1, 2, 4 or 8");
    if (c == 1) mode = TMA_BENCH_UNICAST;
    if (mode < 0 || mode > 2) return bench_fail(GEMM_ERR_INVALID_ARG, "bad mode");
    if (mode != TMA_BENCH_UNICAST && dgc_host::world_is_multi_gpu())
        return bench_fail(GEMM_ERR_UNSUPPORTED, "cluster multicast is single-GPU only; WORLD_SIZE > 1 requires unicast");
    if (o.box_rows < 8 || o.box_rows > 256 || o.box_rows % 8) return bench_fail(GEMM_ERR_UNSUPPORTED, "box_rows 8..256, multiple of 8");
    if (mode == TMA_BENCH_MULTICAST_SLICED && (o.box_rows % (8 * c)))
        return bench_fail(GEMM_ERR_UNSUPPORTED, "sliced multicast needs box_rows a multiple of 8*cluster");
    if (o.stages < 1 || o.stages > 16 || o.iters < 1 || o.warmup < 0 || o.streaming_stride < 0)
        return bench_fail(GEMM_ERR_INVALID_ARG, "stages 1..16, iters >= 1, warmup >= 0, stride >= 0");
    if (cols < 64 || rows < o.box_rows || ld < cols || (ld * 2) % 16 || (reinterpret_cast<uintptr_t>(src) & 15))
        return bench_fail(GEMM_ERR_ALIGNMENT, "src must be 16-byte aligned, ld*2 a multiple of 16, cols >= 64");
    auto enc = encoder();
    if (!enc) return bench_fail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap tm;
    const int box_load_rows = mode == TMA_BENCH_MULTICAST_SLICED ? o.box_rows / c : o.box_rows;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), (cuuint64_t)(((ld * rows * 2) + 15) / 16 * 16)};
    cuuint32_t box[3] = {64, (cuuint32_t)box_load_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(src), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return bench_fail(GEMM_ERR_INVALID_ARG, "tensor map encode failed");
    size_t smem = 1024 + (size_t)o.stages * o.box_rows * 128 + 2 * o.stages * 8;
    if (smem > 232448) return bench_fail(GEMM_ERR_UNSUPPORTED, "stages x tile does not fit in shared memory");
    if (smem < 120 * 1024) smem = 120 * 1024;   // one CTA per SM
    void* fn = reinterpret_cast<void*>(&tma_bench_kernel);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return bench_fail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(64, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int ctas = o.ctas;
    if (ctas <= 0) {
        cfg.gridDim = dim3((unsigned)(sms / c * c), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess || n <= 0) return bench_fail(GEMM_ERR_CUDA, "cudaOccupancyMaxActiveClusters failed");
        ctas = n * c;
    }
    if (ctas % c) return bench_fail(GEMM_ERR_INVALID_ARG, "ctas must be a multiple of cluster");
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    BenchParams p;
    memset(&p, 0, sizeof p);
    p.mode = mode;
    p.cluster = c;
    p.box_rows = o.box_rows;
    p.stages = o.stages;
    p.iters = o.iters;
    p.warmup = o.warmup;
    p.stride = o.streaming_stride;
    p.tiles_x = (int)(cols / 64);
    p.tiles_y = (int)(rows / o.box_rows);
    p.ld = ld;
    p.src = static_cast<const uint16_t*>(src);
    p.cycles = cycles;
    p.ns = ns;
    p.verify = verify;
    p.landed = static_cast<uint8_t*>(o.landed);
    p.origin = o.origin;
    p.timeout_ns = o.wait_timeout_ns ? o.wait_timeout_ns : 2000000000ull;
    void* args[] = {&tm, &p};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return bench_fail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    if (ctas_used) *ctas_used = ctas;
    const double delivered = (double)ctas * o.iters * o.box_rows * 128.0;
    if (delivered_bytes) *delivered_bytes = delivered;
    if (issued_bytes) *issued_bytes = mode == TMA_BENCH_UNICAST ? delivered : delivered / c;
    return GEMM_OK;
}

extern "C" const char* tma_bench_last_error(void) { return g_err; }

extern "C" gemm_status_t tma_bench_query_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return bench_fail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    unsigned int w[4] = {0, 0, 0, 0};
    e = cudaMemcpyFromSymbol(w, g_tma_bench_status, sizeof w);
    if (e != cudaSuccess) return bench_fail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    if (w[0] == 0) return GEMM_OK;
    unsigned int z[4] = {0, 0, 0, 0};
    cudaMemcpyToSymbol(g_tma_bench_status, z, sizeof z);
    snprintf(g_err, sizeof g_err, "tma_bench: bounded wait expired (%s, CTA %u)",
             w[0] == 1 ? "issuer waiting for a free slot" : "consumer waiting for bytes", w[1]);
    return GEMM_ERR_DEVICE_TIMEOUT;
}
