/*
 * stencil.h -- C ABI of the cluster halo-exchange stencil (sm_103a).
 *
 * "集群编程" (cluster programming), sections 分布式共享内存（DSMEM）, 同步 and
 * 实践示例：Halo 交换: the CTAs of a thread-block cluster each hold one tile of
 * a 1-D array in shared memory; after a CTA-wide and then a cluster-wide
 * barrier, a CTA reads its halo elements straight out of its neighbours'
 * shared memory (ld.shared::cluster on a mapa address) instead of going
 * through global memory, and applies the three-point stencil
 *
 *     y[i] = 0.25 * x[i-1] + 0.5 * x[i] + 0.25 * x[i+1]      (x = 0 outside [0, n))
 *
 * Halos that lie in another cluster's tile are read from global memory. A
 * final cluster barrier keeps every CTA alive until its neighbours have read
 * its halo values.
 */
#ifndef STENCIL_H
#define STENCIL_H

#include <stdint.h>
#include "densegemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Elements of x each CTA holds in shared memory (its tile). */
#define STENCIL_TILE 8192

/* y <- stencil(x) for float32 device arrays of n elements, asynchronously on
 * `stream` (a cudaStream_t as void*). cluster: CTAs per cluster, 1, 2, 4 or 8
 * (1 = no DSMEM: every halo comes from global memory). x and y must be 16-byte
 * aligned and must not overlap. n = 0 is a no-op. A bounded wait that expires
 * (the tile load) is reported by stencil_1d_query_status. */
gemm_status_t stencil_1d_run(const float *x, float *y, int64_t n, int cluster, void *stream);

/* Synchronizes `stream`; GEMM_ERR_DEVICE_TIMEOUT if a stencil kernel's wait expired. */
gemm_status_t stencil_1d_query_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* STENCIL_H */
