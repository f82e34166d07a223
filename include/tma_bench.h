/*
 * tma_bench.h -- C ABI of the TMA unicast / multicast load microbenchmark (sm_103a).
 *
 * "Hopper TMA Multicast 深度解析与实测", sections 实测 Microbenchmark 源码 and
 * 实机运行与 NCU 验证: the CTAs of a cluster all need the same 128-byte-wide
 * tile of a bf16 matrix. With unicast every CTA fetches it with its own TMA
 * load; with multicast one load is delivered to every CTA of the cluster, the
 * issuer having armed each receiver's mbarrier with the expected bytes through
 * mapa before issuing. Two scenarios: the same tile over and over (it stays in
 * L2), or a new tile every iteration walking a large matrix (DRAM streaming).
 *
 * One CTA runs per SM (the launch asks for enough shared memory to keep a
 * second one out), so per-CTA rates are per-SM rates.
 *
 * Unlike the page's single-stage loop (one load, a full cluster barrier, the
 * next load), each CTA here keeps `stages` loads in flight in a ring of
 * shared-memory slots guarded by full/empty mbarriers, so the measured rate is
 * the load path's throughput rather than one round trip per load.
 */
#ifndef TMA_BENCH_H
#define TMA_BENCH_H

#include <stdint.h>
#include "densegemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TMA_BENCH_UNICAST = 0,         /* every CTA loads the tile itself */
    TMA_BENCH_MULTICAST = 1,       /* cluster rank 0 loads it once for all (the page's scheme) */
    TMA_BENCH_MULTICAST_SLICED = 2 /* rank r loads rows [r*R/c, (r+1)*R/c) of it for all */
} tma_bench_mode_t;

typedef struct {
    int mode;             /* tma_bench_mode_t */
    int cluster;          /* CTAs per cluster: 1, 2, 4 or 8 (1 forces unicast) */
    int ctas;             /* grid size, a multiple of cluster; 0 = every co-resident cluster */
    int box_rows;         /* rows R per tile (tile = R x 64 bf16 = R x 128 bytes): 8..256, multiple of 8*cluster when sliced */
    int stages;           /* loads in flight per CTA: 1..16 */
    int iters;            /* timed loads per CTA */
    int warmup;           /* untimed loads per CTA before them */
    int streaming_stride; /* 0: every iteration reloads the cluster's own tile (L2-resident);
                             s > 0: iteration i loads tile (i*s*clusters + cluster id) mod tiles */
    uint64_t wait_timeout_ns; /* bound on every in-kernel wait, counted as 2 SM cycles per ns
                                 (this long at 2 GHz, longer at lower clocks); 0 = 2 s */
    void *landed;         /* NULL, or a device array of ctas x box_rows x 128 bytes: after the timed
                             loads each CTA copies its last landed tile there exactly as it sits in
                             shared memory (128-byte swizzle: element (r, j) at byte
                             r*128 + ((j/8) ^ (r%8))*16 + (j%8)*2), for a check of every element */
    int *origin;          /* NULL, or a device array of 2 x ctas ints: that tile's (x, y) origin in src */
} tma_bench_options_t;

/* Runs the benchmark on `stream` (asynchronous) over a rows x cols bf16 matrix
 * `src` (device, row-major, leading dimension ld elements, ld*2 a multiple of 16,
 * cols >= 64). Per CTA it writes:
 *   cycles[i]  -- clock64 cycles of the timed loads (after warmup), CTA i
 *   ns[i]      -- %globaltimer nanoseconds of the same span
 *   verify[i]  -- count of checked elements that did NOT match src (0 = all landed
 *                 where the 128-byte swizzle puts them)
 * Each of cycles, ns, verify is a device array of at least `ctas` entries (the
 * grid size actually used is returned in *ctas_used). Also reports the bytes
 * that land in shared memory (delivered) and that the TMA units fetch (issued):
 * with multicast, issued = delivered / cluster. A bounded wait that expires is
 * reported by tma_bench_query_status. The multicast modes are single-GPU only:
 * with the WORLD_SIZE environment variable above 1 they return
 * GEMM_ERR_UNSUPPORTED before any CUDA call. */
gemm_status_t tma_bench_run(const tma_bench_options_t *opt, const void *src, int64_t rows, int64_t cols,
                            int64_t ld, uint64_t *cycles, uint64_t *ns, uint32_t *verify,
                            int *ctas_used, double *delivered_bytes, double *issued_bytes,
                            void *stream);

/* Synchronizes `stream`; GEMM_ERR_DEVICE_TIMEOUT if a wait of a tma_bench_run
 * kernel expired since the last query, else GEMM_OK. */
gemm_status_t tma_bench_query_status(void *stream);

/* One-line reason for the last failure of a tma_bench_* call on this thread. */
const char *tma_bench_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TMA_BENCH_H */
