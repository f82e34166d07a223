/*
 * densegemm.h -- C ABI of the GB300 (sm_103a) cluster GEMM library.
 *
 * The operation is the tiled dense contraction
 *
 *     C <- alpha * A * B + beta * C          (bf16 A and B, fp32 accumulation,
 *                                             bf16 or fp32 C)
 *
 * and its batched attention-score form S[b] = Q[b] * K[b]^T, which is the same
 * call with B given column-major ("Hopper TMA Multicast 深度解析与实测", section
 * 经典应用场景: S_i = Q_i K^T with the K tile shared by the Q-tile CTAs).
 * How the CTAs of a thread-block cluster share operand tiles is the mode knob:
 *
 *   - unicast: every CTA fetches its own A and B tiles with TMA;
 *   - multicast: one TMA load feeds every CTA of a cluster that needs the same
 *     tile (A along a cluster row, B along a cluster column), the issuer arming
 *     each receiver's mbarrier with the expected bytes through mapa before it
 *     issues ("Hopper TMA Multicast 深度解析与实测", sections 深度机制剖析 and
 *     工程总结; "Clusters, distributed shared memory & cluster launch control",
 *     section "TMA multicast");
 *   - cta_group 2: two CTAs of a cluster run one 256-row tcgen05 MMA, A split by
 *     rows across the pair and B split by columns, each CTA holding its half of
 *     the accumulator in its own tensor memory ("Clusters, distributed shared
 *     memory & cluster launch control", section "Two CTAs, one MMA --
 *     cta_group::2"). It combines with multicast.
 *
 * Work is spread by a persistent, cluster-launched kernel that walks output
 * tiles with a static stride ("Clusters, distributed shared memory & cluster
 * launch control", sections "Thread-block clusters" and "The second wall"),
 * splitting the last waves' k-blocks across clusters (stream-K) or, on request,
 * taking tiles by cluster launch control. Launches carry the programmatic
 * stream serialization attribute: a GEMM may start its prologue while the
 * previous kernel in the stream drains, and waits for it to complete before
 * touching global memory.
 *
 * Conventions for every call:
 *   - Pointers A, B, C are DEVICE pointers owned by the caller (except in
 *     gemm_run_host and gemm_run_strided_batched_host, where they are host
 *     pointers). The library never frees them.
 *   - Sizes and leading dimensions are in elements. A row-major X has its last
 *     index contiguous: element (r, c) at X[r*ld + c]; column-major: X[c*ld + r].
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Runs are asynchronous on it unless a call says otherwise.
 *   - Every call returns a gemm_status_t; nothing exits, aborts or throws across
 *     this boundary. On failure, gemm_last_error() holds a one-line reason.
 *   - A handle is used by one host thread at a time, and its runs must not
 *     overlap on the device: launches of one handle share its stream-K
 *     workspace, tile flags and status word, so runs on different streams need
 *     an ordering between them (an event, or one handle per stream).
 */
#ifndef DENSEGEMM_H
#define DENSEGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_handle_s *gemm_handle_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,    /* a null handle/pointer, negative size, ld too small, bad enum */
    GEMM_ERR_UNSUPPORTED = 2,    /* a mode / cluster / cta_group combination the library does not run */
    GEMM_ERR_ALIGNMENT = 3,      /* a base pointer not 16-byte aligned, or ld/stride bytes not a multiple of 16 */
    GEMM_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed; see gemm_last_error() */
    GEMM_ERR_DEVICE_TIMEOUT = 5, /* a bounded in-kernel wait expired; the kernel stopped cleanly */
    GEMM_ERR_NOT_SM103 = 6       /* the device is not compute capability 10.3 */
} gemm_status_t;

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;
typedef enum { GEMM_OUT_BF16 = 0, GEMM_OUT_F32 = 1 } gemm_out_t;
typedef enum { GEMM_MODE_UNICAST = 0, GEMM_MODE_MCAST = 1 } gemm_mode_t;

/* Test hook: arm 16 bytes more than the first stage will receive, so that the
 * consumer's bounded wait must expire and report GEMM_ERR_DEVICE_TIMEOUT.
 * Nothing faults and nothing spins without a limit. */
#define GEMM_DEBUG_EXTRA_TX 1

typedef struct {
    int mode;           /* gemm_mode_t. UNICAST ignores mcast_a / mcast_b. */
    int mcast_a;        /* 1: multicast each A tile to the CTAs of its cluster row (cluster_n of them) */
    int mcast_b;        /* 1: multicast each B tile to the CTAs of its cluster column
                           (cluster_m of them, or cluster_m / 2 pairs with cta_group 2) */
    int cluster_m;      /* CTAs per cluster along M: 1, 2, 4 or 8 */
    int cluster_n;      /* CTAs per cluster along N: 1, 2, 4 or 8; cluster_m*cluster_n <= 8 */
    int cta_group;      /* 1, 2 for the pair MMA (cluster_m must then be even), or 0: the
                           pair wherever the cluster's extent along M is even (along N for
                           column-major C), else 1; gemm_plan_t.cta_group reports the choice */
    int layout_a;       /* gemm_layout_t of A (M x K) */
    int layout_b;       /* gemm_layout_t of B (K x N) */
    int layout_c;       /* gemm_layout_t of C (M x N) */
    int out_type;       /* gemm_out_t: element type of C */
    int block_n;        /* N extent of one MMA tile: 0 (auto = 256), 128 or 256 */
    int block_k;        /* K extent of one pipeline stage: 0 (auto), 64 or 128; 128 needs K a
                           multiple of 64 when A or B is K-major (auto picks 64 otherwise) */
    int stages;         /* shared-memory pipeline depth; 0 = as many as fit */
    int max_clusters;   /* cap on the persistent grid, in clusters; 0 = as many as are co-resident */
    int group_m;        /* raster band height, in cluster tiles along M; 0 = 4 */
    int schedule;       /* 0 = auto, 1 = whole tiles only, 3 = cluster launch control (one
                           cluster per tile; running clusters cancel pending launches and take
                           their tiles, asking for the next tile before computing the current
                           one), 2 = stream-K: the tiles
                           left after the last full wave (between one and two waves'
                           worth) are split by k-blocks evenly over all clusters, each
                           cluster runs its split pieces before its whole tiles, and the
                           parts are summed in a fixed order; with fewer tiles than
                           clusters, the k-blocks are spread over more clusters (at least
                           16 k-blocks each). Auto splits the tail when that saves at least
                           4 us of an estimated tile time (the tile's FLOPs at 1.5 PFLOP/s
                           shared by all SMs), and spreads a problem with fewer tiles than
                           clusters only when at most half of the clusters would have one.
                           Needs a handle-owned
                           workspace (one 128 x block_n fp32 tile per CTA), so
                           gemm_run_noalloc always runs whole tiles. */
    uint64_t wait_timeout_ns; /* bound on every in-kernel wait, counted as 2 SM cycles per ns
                                 (this long at 2 GHz, longer at lower clocks); 0 = 2 s */
    int debug_flags;    /* 0, or GEMM_DEBUG_EXTRA_TX (tests only) */
    int host_parts;     /* gemm_run_host: parts the problem is split into for overlapping the
                           host copies with the GEMMs, 1 to 8 (fewer when the split dimension
                           is short: parts are multiples of 256 lines); 0 = the count a model
                           of the copy and GEMM times picks */
    int clock_probe;    /* 1: every GEMM launch on this handle adds, per CTA, the SM cycles
                           (clock64) and the %globaltimer nanoseconds from the end of its
                           prologue to its last operand load, and one to a CTA count, to device
                           counters the handle owns, one set per SM (gemm_read_clock sums
                           them): the clock the kernel actually ran at, under load. Two timer
                           reads and three uncontended atomics per CTA, where the issuing
                           thread would wait anyway. 0 = off; gemm_run_noalloc refuses 1. */
} gemm_options_t;

/* What gemm_run would launch for a given problem (host arithmetic only). */
typedef struct {
    int block_m;        /* rows of C per CTA (128) */
    int block_n;        /* columns of C per MMA tile */
    int block_k;        /* K per pipeline stage (64 or 128) */
    int stages;         /* pipeline depth */
    int smem_bytes;     /* dynamic shared memory per CTA */
    int cluster_m, cluster_n;   /* after the column-major-C transpose, if any */
    int cta_group;
    int group_a;        /* CTAs one A fetch serves (1 = unicast) */
    int group_b;        /* CTAs one B fetch serves */
    int transposed;     /* 1: C column-major was computed as C^T = B^T A^T */
    int64_t tiles;      /* cluster tiles in the whole problem (all batches) */
    int64_t clusters;   /* persistent grid size in clusters (before the occupancy cap) */
    int64_t l2_to_sm_operand_bytes; /* analytic TMA operand fetches for the launch */
    int64_t stream_k_tiles;   /* tiles split by k-blocks (0: whole tiles only) */
    int l2_hint_a, l2_hint_b; /* L2 eviction priority of A's / B's loads (the operands as launched,
                                 after the column-major-C transpose): 0 none, 1 evict first (each
                                 tile of it is read by one cluster tile only), 2 evict last (read
                                 by every cluster tile) */
    int k_rotate;             /* 1: whole tiles start their k walk at a tile-dependent k-block */
    int k_serpentine;         /* 1: a cluster's successive whole tiles walk k in alternating directions
                                 and odd raster bands walk their columns from the last (long K, at
                                 least two waves of whole tiles) */
    int prefetch_kb;          /* k-blocks of its first tile each producer prefetches into L2 before
                                 waiting for the previous grid in the stream: the stage count, three
                                 times it on one-tile-wide grids, 0 with cluster launch control */
} gemm_plan_t;

/* Default options: unicast, 1x1 cluster, cta_group 1, A row-major, B column-major,
 * C row-major, bf16 out, everything else automatic. */
void gemm_options_default(gemm_options_t *opt);

/* Checks the options and makes a handle bound to CUDA device `device`.
 * Fails with GEMM_ERR_NOT_SM103 off compute capability 10.3, GEMM_ERR_UNSUPPORTED
 * for an impossible mode (cluster > 8 CTAs, odd cluster_m with cta_group 2, a
 * multicast slice under 8 rows) and for any multicast mode when the environment
 * variable WORLD_SIZE is above 1 (multi-GPU jobs run without cluster multicast).
 * The handle owns a 16-byte device status word and, once needed, the stream-K
 * workspace and the gemm_run_host staging buffers; gemm_destroy frees them.
 * Defined by: the launch set-up of "Clusters, distributed shared memory &
 * cluster launch control", section "Thread-block clusters" (cluster shape as a
 * launch attribute) and the tensor-map descriptors of "Hopper TMA Multicast
 * 深度解析与实测", section 实测 Microbenchmark 源码实现; the mode is fixed here. */
gemm_status_t gemm_create(gemm_handle_t *out, const gemm_options_t *opt, int device);

/* C <- alpha * op(A) * op(B) + beta * C on `stream`, asynchronously.
 * A is M x K with leading dimension lda (layout_a), B is K x N (layout_b), C is
 * M x N (layout_c, out_type). beta == 0 means C is not read (NaN in C does not
 * propagate). M, N or K == 0 is valid: K == 0 gives C <- beta * C.
 * Requirements, checked before any launch: A, B, C 16-byte aligned; lda*2,
 * ldb*2 and ldc*sizeof(C element) multiples of 16 bytes (GEMM_ERR_ALIGNMENT);
 * ld at least the contiguous extent; every dimension below 2^31.
 * Defined by: the contraction itself ("Clusters, distributed shared memory &
 * cluster launch control", section "Where these plug into the GEMM": the tiled
 * GEMM whose CTAs share operand tiles); the operand sharing it runs with is the
 * handle's mode ("Hopper TMA Multicast 深度解析与实测", section 核心架构认知). */
gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda, const void *B, int64_t ldb,
                       void *C, int64_t ldc, float alpha, float beta, void *stream);

/* `batch` independent products C[i] <- alpha*A[i]*B[i] + beta*C[i], where X[i]
 * starts strideX elements after X[i-1]. Strides must be multiples of 16 bytes
 * and keep the matrices apart (at least ld x the stored outer extent), except
 * that strideA or strideB may be 0: one matrix serves every product. Overlapping
 * strides return GEMM_ERR_INVALID_ARG. The attention-score form is
 * A = Q (row-major, sq x d), B = K^T (K given row-major sk x d is B column-major
 * with ldb = d), C = S (fp32, sq x sk).
 * Defined by: "Hopper TMA Multicast 深度解析与实测", section 经典应用场景 (S_i =
 * Q_i K^T for the query tiles of one head, every CTA reading the same K tile). */
gemm_status_t gemm_run_strided_batched(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                       const void *A, int64_t lda, int64_t strideA,
                                       const void *B, int64_t ldb, int64_t strideB,
                                       void *C, int64_t ldc, int64_t strideC, int64_t batch,
                                       float alpha, float beta, void *stream);

/* gemm_run on HOST buffers: copies A, B (and C when beta != 0) to device staging
 * owned by the handle, runs, copies C back, and synchronizes `stream` before
 * returning. The problem is split along the larger of M and N into parts
 * (options.host_parts, or a count a model of the copy and GEMM times picks): the
 * operand every part needs is copied in whole, then part i's slice of the other
 * operand (and of C) is copied in on a handle-owned stream while part i-1 runs
 * on `stream` and part i-2's C is copied out on another, so the copies in both
 * directions overlap each other and the GEMMs. Only the elements of each line
 * are copied (pitched copies): the padding of a leading dimension is neither
 * read nor written on the host. Host buffers may be pageable or pinned; pinned
 * copies are faster and only they overlap. */
gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                            const void *A, int64_t lda, const void *B, int64_t ldb,
                            void *C, int64_t ldc, float alpha, float beta, void *stream);

/* gemm_run_strided_batched on HOST buffers, copied through the handle's staging
 * like gemm_run_host: the batch is split into up to 8 parts of whole products
 * (options.host_parts caps the count), part i's A, B (and C when beta != 0)
 * copied in while part i-1 runs and part i-2's C is copied out. An operand with
 * stride 0 (one matrix for every product) is copied once, first. C comes back line
 * by line unless its batches and lines are
 * dense, so no padding is written on the host. batch = 1 is gemm_run_host.
 * Synchronizes `stream` before returning. */
gemm_status_t gemm_run_strided_batched_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                            const void *A, int64_t lda, int64_t strideA,
                                            const void *B, int64_t ldb, int64_t strideB,
                                            void *C, int64_t ldc, int64_t strideC, int64_t batch,
                                            float alpha, float beta, void *stream);

/* Synchronizes `stream`, then reads and clears the device status word.
 * GEMM_ERR_DEVICE_TIMEOUT if a bounded wait expired in any run since the last
 * query (gemm_last_error() then names the role, stage and CTA).
 * Defined by: "Hopper TMA Multicast 深度解析与实测", section 深度机制剖析 (a
 * receiver's mbarrier waits for bytes another CTA announced; here every such
 * wait is bounded and its expiry is reported instead of hanging). */
gemm_status_t gemm_query_status(gemm_handle_t h, void *stream);

/* Synchronizes `stream`, copies the handle's clock-probe counters to out[0] (SM
 * cycles), out[1] (nanoseconds) and out[2] (CTAs counted), summed over the SMs and the launches
 * since the last read, then clears them; out[0] / out[1] is the mean SM clock in
 * GHz over the CTAs' lifetimes. GEMM_ERR_INVALID_ARG without a handle or out, or
 * for a handle created without options.clock_probe; GEMM_ERR_CUDA if a copy fails.
 * (Measurement plumbing; no page passage.) */
gemm_status_t gemm_read_clock(gemm_handle_t h, void *stream, uint64_t out[3]);

/* Host-only planning: validates `opt` and the problem as gemm_run would and
 * fills `plan`. Needs no GPU; `sm_count` stands in for the device's SM count. */
gemm_status_t gemm_plan(const gemm_options_t *opt, int64_t M, int64_t N, int64_t K,
                        int64_t batch, int sm_count, gemm_plan_t *plan);

/* Static string for a status code. (Library plumbing; no page passage.) */
const char *gemm_status_string(gemm_status_t s);

/* The last failure reason recorded on this handle (or by gemm_create / gemm_plan
 * when h is NULL, per thread). Valid until the next call on the same handle. */
const char *gemm_last_error(gemm_handle_t h);

/* Number of GEMM kernel launches this handle has made (for launch accounting). */
int64_t gemm_launch_count(gemm_handle_t h);

/* gemm_run for callers that cannot allocate device memory. (The pages describe no
 * such entry point; it exists for users of this library.) Some callers must not
 * call cudaMalloc: code running while a memory pool has already reserved the
 * device's memory, allocator callbacks, plugins whose host forbids allocation,
 * or latency-critical paths that cannot afford cudaMalloc's implicit device
 * synchronization. gemm_create allocates a device status record; this call needs
 * no handle and allocates nothing (no cudaMalloc, cudaFree or allocating library
 * routine). Its status record lives in a 256-byte static device array that the
 * library holds on every GPU that loads it until the process exits; a launch
 * uses 16 bytes of it (a size fixed when the library is compiled, and checked
 * against the array's size at compile time). Whole tiles only: the stream-K
 * schedule (schedule 2), which needs a workspace, returns GEMM_ERR_UNSUPPORTED.
 *   - Same arguments and semantics as gemm_create + gemm_run, with the options
 *     and the device given directly; the caller passes A, B and C (device memory).
 *   - The first call on each device does a one-time set-up with that device
 *     current (it looks up the array's device address and the driver's
 *     tensor-map encoder); make that first call before any stream capture.
 *   - Options and sizes are checked before the device is touched; every
 *     argument error returns before anything is enqueued.
 *   - Every call shares the one array and clears the status record on `stream`
 *     right before its GEMM kernel's launch (a call that launches no GEMM kernel,
 *     such as K = 0 or an empty C, leaves it alone). Calls whose kernels overlap
 *     on the GPU race on it, so a timeout seen by one may be reported to another.
 *   - status_out: NULL for a fully asynchronous call; otherwise a host array of
 *     4 uint32 that receives the status record after the call synchronizes
 *     `stream` (GEMM_ERR_DEVICE_TIMEOUT if a bounded wait expired). */
gemm_status_t gemm_run_noalloc(const gemm_options_t *opt, int device, int64_t M, int64_t N, int64_t K,
                               const void *A, int64_t lda, const void *B, int64_t ldb,
                               void *C, int64_t ldc, float alpha, float beta, void *stream,
                               uint32_t *status_out);

/* One unit of a persistent cluster's work (host-only schedule diagnostic). */
typedef struct {
    int64_t tile;          /* cluster tile id (before the raster's mapping to block rows/columns) */
    int32_t kb0, kb1;      /* k-blocks [kb0, kb1) of the tile */
    int32_t kind;          /* 0 whole tile, 1 partial (parks an fp32 partial), 2 finisher */
    int32_t contrib_first; /* finisher: first cluster whose partial it adds (else -1) */
    int32_t contrib_count; /* finisher: number of such clusters, consecutive (else 0) */
    int32_t last;          /* 1 on the cluster's last unit */
} gemm_work_item_t;

/* Host-only: the units cluster `cluster` of a persistent launch walks, in order,
 * for `tiles` cluster tiles of `num_kb` k-blocks on `clusters` clusters, the first
 * `dp_tiles` (a multiple of `clusters` as the planner chooses it) handed out whole
 * by a static stride and the k-blocks of the rest split evenly over all clusters
 * (stream-K, "Clusters, distributed shared memory & cluster launch control",
 * section "The second wall"). The same iterator the kernel runs, compiled for the
 * host. Writes at most `capacity` items and returns how many there are, or -1 for
 * invalid arguments. Needs no GPU. */
int64_t gemm_schedule_work(int64_t tiles, int64_t dp_tiles, int num_kb, int64_t clusters, int64_t cluster,
                           gemm_work_item_t *items, int64_t capacity);

/* Frees the handle and everything it owns. Safe on NULL. (Library plumbing; the
 * kernel-side teardown it pairs with follows "集群编程", section 同步: no CTA
 * leaves while a peer may still address its shared memory.) */
gemm_status_t gemm_destroy(gemm_handle_t h);

#ifdef __cplusplus
}
#endif

#endif /* DENSEGEMM_H */
