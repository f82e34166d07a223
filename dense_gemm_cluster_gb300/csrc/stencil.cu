// Cluster halo-exchange 1-D stencil (see include/stencil.h).
//
// "集群编程", section 实践示例：Halo 交换: each CTA of a cluster loads one tile
// into shared memory, all CTAs meet at a CTA barrier and then a cluster
// barrier (section 同步: write, sync_threads, cluster_sync, read), and each
// reads its left / right halo from its neighbours' shared memory with
// ld.shared::cluster (section 分布式共享内存: the dedicated remote load).
// Here the tile arrives with one bulk asynchronous copy completing on an
// mbarrier, halos across cluster edges come from global memory, and a second
// cluster barrier keeps a CTA's shared memory alive until its neighbours have
// read from it.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "densegemm.h"
#include "ptx.cuh"
#include "stencil.h"

namespace {

constexpr int kThreads = 256;
constexpr int kTile = STENCIL_TILE;
constexpr int kPerThread = kTile / kThreads;         // 32 elements: 8 float4 groups
__device__ unsigned int g_stencil_status[2];

__device__ __forceinline__ float dsmem_load_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__global__ void __launch_bounds__(kThreads)
stencil_1d_kernel(const float* __restrict__ x, float* __restrict__ y, long long n, int cluster) {
    using namespace dgc;
    // data[-1] and data[kTile] hold the halos; data[0] is 16-byte aligned for the bulk copy.
    __shared__ __align__(16) float buf[kTile + 8];
    __shared__ __align__(8) uint64_t bar;
    float* data = buf + 4;
    const int tid = threadIdx.x;
    const uint32_t rank = cluster > 1 ? cluster_ctarank() : 0u;
    const long long start = (long long)blockIdx.x * kTile;
    const long long len_ll = n - start;
    const int len = len_ll <= 0 ? 0 : (len_ll >= kTile ? kTile : (int)len_ll);

    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const uint32_t bulk = (uint32_t)(len * 4) & ~15u;          // whole 16-byte units
        mbar_arrive_expect_tx_local(smem_u32(&bar), bulk);
        if (bulk) bulk_load(smem_u32(data), x + start, bulk, smem_u32(&bar));
        for (int i = (int)(bulk / 4); i < len; ++i) data[i] = x[start + i];   // at most 3 tail elements
        data[len] = 0.0f;                                         // right neighbour past the tile end
        // Bounded wait for the tile (2 SM cycles per ns, 2 s).
        const uint64_t c0 = clock_cycles();
        while (!mbar_try_wait(smem_u32(&bar), 0)) {
            if (clock_cycles() - c0 > 4000000000ull) {
                atomicCAS(&g_stencil_status[0], 0u, 1u);
                g_stencil_status[1] = blockIdx.x;
                break;
            }
        }
    }
    __syncthreads();
    if (cluster > 1) cluster_sync();           // every tile of the cluster is in place

    if (tid == 0 && len > 0) {
        // Left halo: element start-1, the last element of the previous tile.
        float left = 0.0f;
        if (start > 0)
            left = rank > 0 ? dsmem_load_f32(mapa(smem_u32(&data[kTile - 1]), rank - 1)) : x[start - 1];
        // Right halo: element start+len, the first element of the next tile.
        float right = 0.0f;
        if (start + len < n)
            right = rank + 1 < (uint32_t)cluster ? dsmem_load_f32(mapa(smem_u32(&data[0]), rank + 1)) : x[start + len];
        data[-1] = left;
        data[len] = right;
    }
    __syncthreads();

    // Each thread: 8 groups of 4 consecutive elements, groups 1024 elements apart.
#pragma unroll
    for (int g = 0; g < kPerThread / 4; ++g) {
        const int e = g * (kThreads * 4) + tid * 4;
        if (e + 3 < len) {
            float4 o;
            o.x = 0.25f * data[e - 1] + 0.5f * data[e] + 0.25f * data[e + 1];
            o.y = 0.25f * data[e] + 0.5f * data[e + 1] + 0.25f * data[e + 2];
            o.z = 0.25f * data[e + 1] + 0.5f * data[e + 2] + 0.25f * data[e + 3];
            o.w = 0.25f * data[e + 2] + 0.5f * data[e + 3] + 0.25f * data[e + 4];
            *reinterpret_cast<float4*>(y + start + e) = o;
        } else {
            for (int q = 0; q < 4 && e + q < len; ++q)
                y[start + e + q] = 0.25f * data[e + q - 1] + 0.5f * data[e + q] + 0.25f * data[e + q + 1];
        }
    }
    if (cluster > 1) cluster_sync();           // neighbours are done reading this CTA's halo values
}

thread_local char g_stencil_err[256];

gemm_status_t sfail(gemm_status_t s, const char* m) {
    snprintf(g_stencil_err, sizeof g_stencil_err, "%s", m);
    return s;
}

}  // namespace

extern "C" gemm_status_t stencil_1d_run(const float* x, float* y, int64_t n, int cluster, void* stream) {
    if (n < 0) return sfail(GEMM_ERR_INVALID_ARG, "negative n");
    if (n == 0) return GEMM_OK;
    if (!x || !y) return sfail(GEMM_ERR_INVALID_ARG, "null pointer");
    if (cluster != 1 && cluster != 2 && cluster != 4 && cluster != 8)
        return sfail(GEMM_ERR_UNSUPPORTED, "cluster must be 1, 2, 4 or 8");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return sfail(GEMM_ERR_ALIGNMENT, "x and y must be 16-byte aligned");
    const char* xb = reinterpret_cast<const char*>(x);
    const char* yb = reinterpret_cast<const char*>(y);
    if (xb < yb + n * 4 && yb < xb + n * 4) return sfail(GEMM_ERR_INVALID_ARG, "x and y overlap");
    long long tiles = (n + kTile - 1) / kTile;
    tiles = (tiles + cluster - 1) / cluster * cluster;   // whole clusters; extra CTAs hold no elements
    if (tiles >= (1ll << 31)) return sfail(GEMM_ERR_INVALID_ARG, "n too large");
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)tiles, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, stencil_1d_kernel, x, y, (long long)n, cluster);
    if (e != cudaSuccess) return sfail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    return GEMM_OK;
}

extern "C" gemm_status_t stencil_1d_query_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return sfail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    unsigned int w[2] = {0, 0};
    e = cudaMemcpyFromSymbol(w, g_stencil_status, sizeof w);
    if (e != cudaSuccess) return sfail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    if (w[0] == 0) return GEMM_OK;
    unsigned int z[2] = {0, 0};
    cudaMemcpyToSymbol(g_stencil_status, z, sizeof z);
    return sfail(GEMM_ERR_DEVICE_TIMEOUT, "stencil: the tile load did not complete");
}
