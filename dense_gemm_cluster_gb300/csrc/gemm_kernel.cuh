// Persistent, cluster-launched, warp-specialised GEMM for sm_103a.
//
//   C[b] <- alpha * A[b] * B[b] + beta * C[b]      bf16 A/B, fp32 accumulate in TMEM
//
// One CTA owns 128 rows of C (BLOCK_M). A cluster of cx * cy CTAs (cx along M,
// cy along N) covers a "cluster tile" of cx*128 rows by cy*BN columns. Roles:
//
//   warp 0      A producer: TMA loads of A k-blocks into an S-stage ring
//   warp 6      B producer: the same for B (two issuing threads keep the TMA
//               engine fed: one thread's arm/issue/wait latency per k-block is
//               longer than the tensor core's time for it)
//   warp 1      TMEM allocation; MMA issue (one elected lane; with the pair MMA
//               only the pair's even CTA issues)
//   warps 2..5  epilogue: TMEM -> registers -> (alpha, beta) -> shared -> TMA store
//
// Operand sharing ("Hopper TMA Multicast 深度解析与实测", sections
// 核心架构认知 / 深度机制剖析 / 工程总结; "Clusters, distributed shared memory &
// cluster launch control", sections "TMA multicast" and "Two CTAs, one MMA"):
//   * A multicast: the cy CTAs of a cluster row share A. CTA with row index
//     idxA loads rows [idxA*128/cy, (idxA+1)*128/cy) of the A tile and delivers
//     them to every CTA of the row with one multicast.
//   * B multicast: the CTAs of a cluster column that hold the same B columns
//     (all cx of them, or the cx/2 CTAs of equal parity with the pair MMA)
//     split and multicast the B tile the same way.
//   * Before each load the issuer arms, for every receiving CTA, the barrier
//     that will count those bytes (its own or a peer's, through mapa), so no
//     barrier can complete before every delivery it waits for is announced.
//   * Pair MMA (G = 2): CTAs 2p and 2p+1 of a cluster column form a pair; the
//     even CTA issues tcgen05.mma.cta_group::2 with M = 256 (A rows split across
//     the pair) and N = BN (B columns split across the pair). Every TMA load of
//     the pair signals the even CTA's barrier.
//   * Stage reuse: each consumer commits its release of stage s to the "empty"
//     barrier of every CTA that writes into its shared memory, so an issuer
//     only overwrites a stage once all its receivers are done with it.
//
// Tile order is a static persistent stride over cluster tiles ("Clusters,
// distributed shared memory & cluster launch control", section "The second
// wall"), rastered in bands of group_m cluster-rows so that co-running
// clusters share A and B tiles in L2 (with the serpentine walk, odd bands walk
// their columns from the last). The tiles after the last full wave may be split
// by k-blocks evenly over all clusters (stream-K: each cluster runs its pieces
// before its whole tiles; the piece holding a tile's first k-block adds the
// others' fp32 partials in cluster order, so the sum is deterministic). With
// cluster launch control every tile is its own cluster launch, and running
// clusters cancel pending ones and take their tiles (section "Cluster launch
// control").
//
// L2 traffic: when the tile grid is one tile wide, the operand that each tile
// reads alone is loaded with an evict-first policy and the one every tile reads
// with evict-last (K-major streamed rows also start at a tile-dependent k-block);
// on long-K grids of several waves a cluster's successive whole tiles, which share
// their A rows in the raster band, walk k in alternating directions, so each
// starts on the k-blocks L2 received last; each producer prefetches the first
// k-blocks of its first tile into L2 before waiting for the previous grid in the
// stream (programmatic dependent launch), deeper than the ring on one-tile-wide grids.
//
// Every wait is bounded by wait_timeout_ns of %globaltimer; on expiry the
// thread records a status word in global memory, raises a CTA-wide abort flag
// and its role stops, so the kernel always returns.
//
// Clock probe (optional): the A producer adds its CTA's SM cycles and
// %globaltimer nanoseconds, from the end of the prologue to its last load, to
// its SM's slot of a counter buffer: the clock the kernel ran at.
#pragma once
#include <cuda.h>
#include <cstdint>
#include "ptx.cuh"

namespace dgc {

constexpr int BLOCK_M = 128;
constexpr int ATOM_K = 64;                                       // bf16 elements per 128-byte swizzle row
constexpr int NUM_THREADS = 224;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF_BYTES = 4096;                              // 32 rows x 128 bytes
constexpr int EPI_SMEM_BYTES = EPI_WARPS * 2 * EPI_BUF_BYTES;    // double-buffered per warp

// Error codes written to status[0] by a wait that ran out.
enum : uint32_t {
    ERR_NONE = 0,
    ERR_WAIT_EMPTY = 1,      // producer waiting for a stage to be released
    ERR_WAIT_FULL = 2,       // MMA waiting for a stage's bytes
    ERR_WAIT_TMEM_EMPTY = 3, // MMA waiting for the epilogue to free an accumulator
    ERR_WAIT_TMEM_FULL = 4,  // epilogue waiting for an accumulator
    ERR_WAIT_DRAIN = 5,      // teardown waiting for in-flight MMAs
    ERR_WAIT_PARTIAL = 6,    // stream-K finisher waiting for another cluster's partial
    ERR_WAIT_TILE_ID = 7,    // a role waiting for the next tile from cluster launch control
    ERR_WAIT_TILE_SLOT = 8,  // the scheduler waiting for a free tile-id slot
    ERR_WAIT_FIXUP = 9,      // stream-K finisher waiting for partials copied into shared memory
};

constexpr int TILE_RING = 4;   // cluster-launch-control responses in flight per cluster
constexpr int CLOCK_PROBE_SLOTS = 256;   // per-SM counter slots of the clock probe (%smid modulo this)

struct KernelParams {
    int M, N, K;             // problem (after any transpose for column-major C)
    int batch;
    int num_kb;              // ceil(K / BK), >= 1
    int a_kmap4, b_kmap4;    // K-major operand described by the 4-D k-split map {64, rows, K/64, batch}
    int cx, cy;              // cluster extent along M / N (CTAs)
    int mcast_a, mcast_b;
    int a_mn_major, b_mn_major;
    int out_f32;
    int tiles_m, tiles_n;    // cluster tiles along M / N per batch
    long long total_tiles;   // tiles_m * tiles_n * batch
    int group_m;
    int stages;
    int debug_flags;
    float alpha, beta;
    const void* c_in;        // C (read when beta != 0)
    long long ldc, stride_c; // elements
    unsigned int* status;    // 4 words: code, detail, block, tile
    unsigned long long timeout_ns;
    // Stream-K split: tiles [0, dp_tiles) go whole to clusters by a static stride;
    // the sk_iters k-blocks of the remaining tiles are split evenly over the clusters
    // (each cluster runs its split pieces before its whole tiles).
    long long dp_tiles;
    long long sk_iters;
    float* workspace;        // one BLOCK_M x BN fp32 partial slot per CTA of the grid
    unsigned int* flags;     // per slot: 1 while the slot holds a partial not yet summed, else 0
    int clc;                 // 1: one cluster per tile; running clusters take pending ones' tiles
    int a_shared, b_shared;  // 1: one matrix serves every product of the batch (stride 0)
    int a_l2, b_l2;          // L2 eviction priority of the operand's loads: 0 none, 1 evict first, 2 evict last
    int k_rotate;            // 1: whole tiles start their k walk at a tile-dependent k-block
    int k_serpentine;        // 1: a cluster's successive whole tiles alternate their k direction
    int prefetch_kb;         // k-blocks of the first tile prefetched into L2 before waiting for the previous grid
    unsigned long long* clk; // clock probe: CLOCK_PROBE_SLOTS x (cycles, ns, CTAs), or null
};

enum : int { L2_HINT_NONE = 0, L2_HINT_EVICT_FIRST = 1, L2_HINT_EVICT_LAST = 2 };

struct TileCoord {
    int b, ctm, ctn;
};

__host__ __device__ __forceinline__ TileCoord tile_coord(const KernelParams& p, long long t) {
    const long long per_batch = (long long)p.tiles_m * p.tiles_n;
    TileCoord c;
    c.b = (int)(t / per_batch);
    const long long r = t - (long long)c.b * per_batch;
    const long long in_group = (long long)p.group_m * p.tiles_n;
    const int group = (int)(r / in_group);
    const int first_m = group * p.group_m;
    const int gsz = p.group_m < p.tiles_m - first_m ? p.group_m : p.tiles_m - first_m;
    const int local = (int)(r - (long long)group * in_group);
    c.ctm = first_m + local % gsz;
    c.ctn = local / gsz;
    // With the serpentine walk the bands snake too: odd bands walk their columns from the
    // last, so a band starts on the B columns the previous band read last.
    if (p.k_serpentine && (group & 1)) c.ctn = p.tiles_n - 1 - c.ctn;
    return c;
}

// One unit of work of a cluster: k-blocks [kb0, kb1) of cluster tile `tile`.
//   WHOLE:    the full K range; the epilogue stores C.
//   PARTIAL:  a later part of a tile whose first k-block another cluster owns;
//             the epilogue writes the fp32 partial to this CTA's workspace slot
//             and raises its flag.
//   FINISHER: the first part of a tile whose rest other clusters compute; the
//             epilogue adds their partials (in cluster order) before storing C,
//             then lowers their flags, so every launch starts with all flags down
//             and the kernel carries no per-launch host state (a CUDA graph can
//             replay it).
enum : int { WORK_WHOLE = 0, WORK_PARTIAL = 1, WORK_FINISHER = 2 };

struct Work {
    long long tile;
    int kb0, kb1;
    int kind;
    int contrib_first, contrib_count;   // FINISHER: clusters whose slots hold the rest
    bool last;                          // the cluster's last work item (no load follows it)
};

// Cluster launch control ("Clusters, distributed shared memory & cluster launch
// control", sections "Cluster launch control" and "The work-stealing loop"):
// the grid has one cluster per tile; a running cluster asks the hardware to
// cancel a not-yet-launched cluster and takes its tile. The request for the
// next tile goes out before the current tile is computed; the loop ends when a
// request comes back not canceled (there is no sentinel tile id). Responses
// land in a small ring in every CTA of the cluster; every role reads them.
struct ClcCtx {
    uint32_t resp0;          // shared address of response slot 0 (16 bytes each)
    uint32_t full0;          // ring "response landed" barriers (8 bytes each)
    uint32_t empty_rank0;    // rank 0's ring "slot read by everyone" barrier 0, as a cluster address
    uint32_t cs;             // CTAs per cluster
    volatile int* abort_flag;
    int consumed;            // ring entries read so far
    bool arrive;             // this thread reports its reads (one thread per role)
};

__device__ bool clc_next(const KernelParams& p, ClcCtx& c, long long& tile);

// Static persistent schedule with a stream-K split ("Clusters, distributed
// shared memory & cluster launch control", section "The second wall": a fixed
// stride leaves SMs idle in the last wave when tiles do not divide evenly;
// splitting the last waves' k-blocks evenly over all clusters removes that
// idle time). Every role of every CTA of a cluster walks the same sequence.
// Compiled for the host too, where gemm_schedule_work replays it so that the
// partition can be checked without a GPU.
struct WorkIter {
    long long dp_next, sk_it, sk_end, cid, ncl, base, rem;
    ClcCtx* clc = nullptr;   // set: tiles come from cluster launch control
    bool first_done = false;

    __host__ __device__ void init(const KernelParams& p, long long cluster, long long clusters,
                                  ClcCtx* ctx = nullptr) {
        clc = p.clc ? ctx : nullptr;
        first_done = false;
        cid = cluster;
        ncl = clusters;
        dp_next = cluster;
        base = p.sk_iters / clusters;
        rem = p.sk_iters % clusters;
        sk_it = start_of(cluster);
        sk_end = start_of(cluster + 1);
    }
    __host__ __device__ long long start_of(long long c) const { return c * base + (c < rem ? c : rem); }

    // The stream-K pieces come first and the whole tiles after them, so a finisher's
    // wait for its contributors' partials and its fixup overlap the whole tiles'
    // mainloops instead of ending the kernel. A contributor's piece is always the
    // first of its range, so every partial is parked at the start.
    __host__ __device__ bool next(const KernelParams& p, Work& w) {
        if (clc) {
            long long t = cid;                  // the first tile is this cluster's own
#ifdef __CUDA_ARCH__
            if (first_done && !clc_next(p, *clc, t)) return false;
#else
            if (first_done) return false;       // cluster launch control has no host form
#endif
            first_done = true;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.num_kb;
            w.kind = WORK_WHOLE;
            w.last = false;
            return true;
        }
        if (sk_it >= sk_end) {
            if (dp_next >= p.dp_tiles) return false;
            w.tile = dp_next;
            w.kb0 = 0;
            w.kb1 = p.num_kb;
            w.kind = WORK_WHOLE;
            dp_next += ncl;
            w.last = dp_next >= p.dp_tiles;
            return true;
        }
        const long long rel = sk_it / p.num_kb;
        w.tile = p.dp_tiles + rel;
        w.kb0 = (int)(sk_it - rel * p.num_kb);
        const long long left = sk_end - sk_it;
        w.kb1 = (int)((long long)(p.num_kb - w.kb0) < left ? p.num_kb : w.kb0 + left);
        if (w.kb0 > 0) {
            w.kind = WORK_PARTIAL;
        } else if (w.kb1 < p.num_kb) {
            w.kind = WORK_FINISHER;
            const long long tile_end = (rel + 1) * p.num_kb;
            w.contrib_first = (int)(cid + 1);
            int n = 0;
            while (cid + 1 + n < ncl && start_of(cid + 1 + n) < tile_end) ++n;
            w.contrib_count = n;
        } else {
            w.kind = WORK_WHOLE;
        }
        sk_it += w.kb1 - w.kb0;
        w.last = sk_it >= sk_end && dp_next >= p.dp_tiles;
        return true;
    }
};

__device__ __noinline__ void report_timeout(const KernelParams& p, uint32_t code, uint32_t detail,
                                            long long tile) {
    if (atomicCAS(p.status, 0u, code) == 0u) {
        p.status[1] = detail;
        p.status[2] = blockIdx.x;
        p.status[3] = (unsigned int)tile;
        __threadfence();
    }
}

// Bounded wait on phase `parity` of the barrier at `bar`. Returns false (after
// recording the reason unless another role already aborted) when the budget is
// spent or the CTA is aborting.
template <bool CLUSTER_SCOPE = false>
__device__ __forceinline__ bool probe(uint32_t bar, uint32_t parity) {
    return CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

template <bool CLUSTER_SCOPE = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const KernelParams& p,
                                             volatile int* abort_flag, uint32_t code, uint32_t detail,
                                             long long tile) {
    if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
    // The budget is counted in SM cycles (cheap to read) at 2 cycles per ns:
    // at most twice the nominal time at the maximum clock, longer when slower.
    const uint64_t c0 = clock_cycles();
    const uint64_t budget = 2ull * p.timeout_ns;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (probe<CLUSTER_SCOPE>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock_cycles() - c0 > budget) {
            report_timeout(p, code, detail, tile);
            *abort_flag = 1;
            return false;
        }
    }
}

// Reads the next cluster-launch-control response: false when the request was
// not canceled (no tile left) or the wait ran out.
__device__ bool clc_next(const KernelParams& p, ClcCtx& c, long long& tile) {
    const int slot = c.consumed % TILE_RING;
    const uint32_t phase = (uint32_t)(c.consumed / TILE_RING) & 1u;
    if (!wait_bounded(c.full0 + 8u * slot, phase, p, c.abort_flag, ERR_WAIT_TILE_ID, (uint32_t)slot, -1))
        return false;
    uint32_t x = 0;
    const bool got = clc_decode(c.resp0 + 16u * slot, &x);
    if (c.arrive) mbar_arrive_cluster(c.empty_rank0 + 8u * slot);
    ++c.consumed;
    if (!got) return false;
    tile = (long long)(x / c.cs);
    return true;
}

// Bitmask of the CTAs of cluster row `rx` (same A rows), ranks rx + cx*y.
__device__ __forceinline__ uint32_t row_mask(int rx, int cx, int cy) {
    uint32_t m = 0;
    for (int y = 0; y < cy; ++y) m |= 1u << (rx + cx * y);
    return m;
}
// Bitmask of the CTAs of cluster column `ry` holding the same B columns:
// every x (G = 1) or every x of the same parity as rx (G = 2).
template <int G>
__device__ __forceinline__ uint32_t col_mask(int rx, int ry, int cx) {
    uint32_t m = 0;
    for (int x = (G == 2 ? (rx & 1) : 0); x < cx; x += G) m |= 1u << (x + cx * ry);
    return m;
}

// Whole tiles may start their k walk at a tile-dependent k-block (wrapping around),
// so that concurrent tiles do not all ask L2 for the same k-block of the operand they
// share. Returns the offset for work `w` (0: in order).
__device__ __forceinline__ int k_rotation(const KernelParams& p, const Work& w) {
    const int nkb = w.kb1 - w.kb0;
    if (!p.k_rotate || w.kind != WORK_WHOLE || nkb < 2) return 0;
    const long long t = w.tile;
    return (int)(((t * (long long)nkb) / (p.total_tiles > 0 ? p.total_tiles : 1) + t) % nkb);
}

// One operand's producer loop (run by one thread). Per k-block (BK wide): wait
// until the stage is released by every CTA this thread writes into, arm each
// receiver's full barrier with the bytes of this thread's slice (through mapa
// for peers), then issue the slice, multicast when it feeds several CTAs.
// Shared-memory tile layouts (128-byte swizzle throughout):
//   K-major (rows x BK): BK/64 atoms, each rows x 128 bytes, atom after atom.
//     With the 4-D k-split map one load fills any run of whole atoms, so a
//     group of `parts` issuers splits the tile by atoms first (parts <= BK/64)
//     and then by rows within an atom: one TMA load per issuer per stage.
//     Without it (K not a multiple of 64; BK = 64) a slice is a band of rows.
//   MN-major (BK x rows): rows/64 boxes of BK K-rows x 128 bytes; a slice is a
//     band of K rows of every box (one TMA load per box).
struct OperandPlan {
    const CUtensorMap* tmap;
    uint32_t tile0;        // shared address of stage 0's tile
    uint32_t tile_bytes;   // per stage
    int rows;              // MN extent of the tile held by this CTA
    int mn_major;
    int kmap4;             // K-major with the 4-D k-split map
    int slice, parts;      // this CTA's slice index and the group size
    uint32_t mask;         // receivers (multicast) or just this CTA
    int shared;            // one matrix for the whole batch: batch coordinate 0
};

template <int G, int BK, bool HINT>
__device__ __forceinline__ void tma_issue(const OperandPlan& op, bool mcast, uint32_t dst, uint32_t bar, int x, int y,
                                          int z, int w, bool four_d, uint64_t pol) {
    if constexpr (HINT) {
        if (four_d) {
            if (G == 1) {
                if (mcast) tma_load_4d_mcast_hint(dst, op.tmap, bar, x, y, z, w, (uint16_t)op.mask, pol);
                else       tma_load_4d_hint(dst, op.tmap, bar, x, y, z, w, pol);
            } else {
                if (mcast) tma_load_4d_pair_mcast_hint(dst, op.tmap, bar, x, y, z, w, (uint16_t)op.mask, pol);
                else       tma_load_4d_pair_hint(dst, op.tmap, bar, x, y, z, w, pol);
            }
        } else {
            if (G == 1) {
                if (mcast) tma_load_3d_mcast_hint(dst, op.tmap, bar, x, y, z, (uint16_t)op.mask, pol);
                else       tma_load_3d_hint(dst, op.tmap, bar, x, y, z, pol);
            } else {
                if (mcast) tma_load_3d_pair_mcast_hint(dst, op.tmap, bar, x, y, z, (uint16_t)op.mask, pol);
                else       tma_load_3d_pair_hint(dst, op.tmap, bar, x, y, z, pol);
            }
        }
    } else {
    if (four_d) {
        if (G == 1) {
            if (mcast) tma_load_4d_mcast(dst, op.tmap, bar, x, y, z, w, (uint16_t)op.mask);
            else       tma_load_4d(dst, op.tmap, bar, x, y, z, w);
        } else {
            if (mcast) tma_load_4d_pair_mcast(dst, op.tmap, bar, x, y, z, w, (uint16_t)op.mask);
            else       tma_load_4d_pair(dst, op.tmap, bar, x, y, z, w);
        }
    } else {
        if (G == 1) {
            if (mcast) tma_load_3d_mcast(dst, op.tmap, bar, x, y, z, (uint16_t)op.mask);
            else       tma_load_3d(dst, op.tmap, bar, x, y, z);
        } else {
            if (mcast) tma_load_3d_pair_mcast(dst, op.tmap, bar, x, y, z, (uint16_t)op.mask);
            else       tma_load_3d_pair(dst, op.tmap, bar, x, y, z);
        }
    }
    }
}

// This issuer's part of a stage's tile (see the layouts above).
struct SliceGeom {
    int atom0, r0, k_rows;
    uint32_t slice_off;      // byte offset of the part within the tile
};

template <int BK>
__device__ __forceinline__ SliceGeom slice_geom(const OperandPlan& op) {
    constexpr int NAT = BK / ATOM_K;
    SliceGeom g{0, 0, BK, 0u};
    if (op.mn_major) {
        g.k_rows = BK / op.parts;
        g.slice_off = (uint32_t)(op.slice * g.k_rows * 128);
    } else if (op.kmap4) {
        if (op.parts <= NAT) {
            g.atom0 = op.slice * (NAT / op.parts);
        } else {
            const int rparts = op.parts / NAT;
            g.atom0 = op.slice / rparts;
            g.r0 = (op.slice % rparts) * (op.rows / rparts);
        }
        g.slice_off = (uint32_t)(g.atom0 * op.rows * 128 + g.r0 * 128);
    } else {
        g.r0 = op.slice * (op.rows / op.parts);
        g.slice_off = (uint32_t)(g.r0 * 128);
    }
    return g;
}

// Prefetches into L2 this issuer's part of the first `nkb_max` k-blocks of its cluster's
// first work item: the same boxes produce() will load, so a launch that follows another in
// the stream overlaps its first DRAM reads with the previous grid's last tiles. A
// prefetch returns no data to the SM, so it may run before griddepcontrol.wait.
template <int G, int BK>
__device__ __forceinline__ void prefetch_first_stages(const KernelParams& p, const OperandPlan& op, bool is_a, int cx,
                                                      int cy, int rx, int ry, int BNv, int BN_CTAv, long long cluster,
                                                      long long clusters, int nkb_max) {
    constexpr int NAT = BK / ATOM_K;
    WorkIter wi;
    wi.init(p, cluster, clusters, nullptr);
    Work w;
    if (!wi.next(p, w)) return;
    const SliceGeom sg = slice_geom<BK>(op);
    const TileCoord tc = tile_coord(p, w.tile);
    const int zb = op.shared ? 0 : tc.b;
    const int mn0 = is_a ? (tc.ctm * cx + rx) * BLOCK_M
                         : (tc.ctn * cy + ry) * BNv + (G == 2 ? (rx & 1) * BN_CTAv : 0);
    const int nkb = w.kb1 - w.kb0;
    const int rot = k_rotation(p, w);
    for (int i = 0; i < nkb_max && i < nkb; ++i) {
        const int kb = w.kb0 + (i + rot < nkb ? i + rot : i + rot - nkb);
        if (op.mn_major) {
            const int y = kb * BK + op.slice * sg.k_rows;
            for (int box = 0; box < op.rows / 64; ++box) tma_prefetch_3d(op.tmap, mn0 + box * 64, y, zb);
        } else if (op.kmap4) {
            tma_prefetch_4d(op.tmap, 0, mn0 + sg.r0, kb * NAT + sg.atom0, zb);
        } else {
            tma_prefetch_3d(op.tmap, kb * BK, mn0 + sg.r0, zb);
        }
    }
}

// WALK_PLAIN: k-blocks in order, no hints. WALK_ONE_WIDE: the planner's one-tile-wide
// grid policy (L2 eviction priorities and, when set, the rotated k walk). WALK_SERPENTINE:
// whole tiles alternate their k direction from one of a cluster's tiles to the next, so
// each starts on the k-blocks its predecessor read last.
enum : int { WALK_PLAIN = 0, WALK_ONE_WIDE = 1, WALK_SERPENTINE = 2 };

template <int G, int BK, int WALK>
__device__ __forceinline__ bool produce(const KernelParams& p, const OperandPlan& op, bool is_a, uint32_t full0,
                                        uint32_t empty0, uint32_t rank, uint32_t leader, int cx, int cy, int rx,
                                        int ry, int BNv, int BN_CTAv, volatile int* abort_flag,
                                        long long cluster, long long clusters, int S, ClcCtx* clc,
                                        uint32_t ring_empty0) {
    constexpr int NAT = BK / ATOM_K;             // swizzle atoms per stage along K
    // Arm targets: the barrier that counts each receiver's bytes (the receiver
    // itself, or its pair's even CTA), resolved once and indexed by receiver
    // rank with compile-time indices so the table stays in registers.
    uint32_t arm_addr[8];
#pragma unroll
    for (int d = 0; d < 8; ++d)
        arm_addr[d] = (op.mask & (1u << d)) ? mapa(full0, G == 2 ? ((uint32_t)d & ~1u) : (uint32_t)d) : 0u;
    const uint32_t slice_bytes = op.tile_bytes / (uint32_t)op.parts;
    const uint32_t tma_bar0 = (G == 2) ? mapa(full0, leader) : full0;
    const bool mcast = op.parts > 1;
    const SliceGeom sg = slice_geom<BK>(op);
    bool extra_tx = is_a && (p.debug_flags & 1) != 0;
    // L2 eviction priority of this operand's loads (chosen by the planner).
    constexpr bool HINTED = WALK == WALK_ONE_WIDE;
    uint64_t pol = 0;
    if constexpr (HINTED) {
        const int l2 = is_a ? p.a_l2 : p.b_l2;
        pol = l2 == L2_HINT_EVICT_FIRST ? l2_policy_evict_first() : l2_policy_evict_last();
    }
    int stage = 0;
    uint32_t phase = 0;
    WorkIter wi;
    wi.init(p, cluster, clusters, clc);
    Work w;
    const bool scheduler = p.clc && is_a && rank == 0;
    int requests = 0;
    while (wi.next(p, w)) {
        const long long t = w.tile;
        if (scheduler) {
            // Ask for the next tile before computing this one.
            const int slot = requests % TILE_RING;
            const uint32_t ph = (uint32_t)(requests / TILE_RING) & 1u;
            if (!wait_bounded<true>(ring_empty0 + 8u * slot, ph ^ 1u, p, abort_flag, ERR_WAIT_TILE_SLOT,
                                    (uint32_t)slot, t))
                return false;
            for (uint32_t r = 0; r < clc->cs; ++r)
                mbar_arrive_expect_tx_cluster(mapa(clc->full0 + 8u * slot, r), 16u);
            clc_try_cancel(clc->resp0 + 16u * slot, clc->full0 + 8u * slot, clc->cs > 1);
            ++requests;
        }
        const TileCoord tc = tile_coord(p, t);
        const int zb = op.shared ? 0 : tc.b;           // batch coordinate of this operand
        const int mn0 = is_a ? (tc.ctm * cx + rx) * BLOCK_M
                             : (tc.ctn * cy + ry) * BNv + (G == 2 ? (rx & 1) * BN_CTAv : 0);
        const int nkb = w.kb1 - w.kb0;
        const int rot = WALK == WALK_ONE_WIDE ? k_rotation(p, w) : 0;
        const bool back = WALK == WALK_SERPENTINE && w.kind == WORK_WHOLE && ((w.tile / clusters) & 1);
        for (int i = 0; i < nkb; ++i) {
            const int kb = WALK == WALK_ONE_WIDE ? w.kb0 + (i + rot < nkb ? i + rot : i + rot - nkb)
                         : WALK == WALK_SERPENTINE ? (back ? w.kb1 - 1 - i : w.kb0 + i)
                                                   : w.kb0 + i;
            if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, p, abort_flag, ERR_WAIT_EMPTY, (uint32_t)stage, t))
                return false;
#pragma unroll
            for (int d = 0; d < 8; ++d)
                if (op.mask & (1u << d)) mbar_arrive_expect_tx_cluster(arm_addr[d] + 8u * stage, slice_bytes);
            if (extra_tx) {
                // Test hook: announce bytes that never come; the MMA's bounded
                // wait on this stage must run out.
                asm volatile("mbarrier.expect_tx.relaxed.cluster.shared::cluster.b64 [%0], %1;"
                             :: "r"(mapa(full0 + 8u * stage, leader)), "r"(16u) : "memory");
                extra_tx = false;
            }
            const uint32_t bar = tma_bar0 + 8u * stage;
            const uint32_t dst = op.tile0 + stage * op.tile_bytes + sg.slice_off;
            if (op.mn_major) {
                const int y = kb * BK + op.slice * sg.k_rows;
                for (int box = 0; box < op.rows / 64; ++box)
                    tma_issue<G, BK, HINTED>(op, mcast, dst + (uint32_t)(box * BK * 128), bar, mn0 + box * 64, y, zb,
                                             0, false, pol);
            } else if (op.kmap4) {
                tma_issue<G, BK, HINTED>(op, mcast, dst, bar, 0, mn0 + sg.r0, kb * NAT + sg.atom0, zb, true, pol);
            } else {
                tma_issue<G, BK, HINTED>(op, mcast, dst, bar, kb * BK, mn0 + sg.r0, zb, 0, false, pol);
            }
            if (++stage == S) { stage = 0; phase ^= 1u; }
        }
    }
    // Drain: every stage this thread filled is released by all its receivers
    // before the CTA may exit (no remote arrival may target an exited CTA).
    for (int i = 0; i < S; ++i) {
        if (!wait_bounded(empty0 + 8u * stage, phase ^ 1u, p, abort_flag, ERR_WAIT_EMPTY, (uint32_t)stage, -1))
            return false;
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
    return true;
}

// Where a stream-K finisher's epilogue warp stages the partials it adds: its
// quarter of the operand ring, free once the finisher's last MMA has completed
// when the finisher is the cluster's last work item (no load lands there any
// more), filled by bulk copies that complete on the warp's own barrier. A
// finisher followed by whole tiles stages nothing (bytes = 0) and adds the
// partials from global memory while the ring refills.
struct FixStage {
    uint8_t* ptr;        // generic address of the warp's region
    uint32_t saddr;      // its shared-memory address
    uint32_t bytes;      // region size
    uint32_t bar;        // the warp's barrier
    uint32_t* phase;     // its next phase
    volatile int* abort_flag;
};

__device__ __forceinline__ void bulk_load_smem(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// One epilogue warp's rows of one output tile.
struct EpiTile {
    uint32_t t_row;      // TMEM address of this warp's lanes, this accumulator's column 0
    int n0;              // first column of the tile
    int row0;            // first global row this warp stores (32 rows)
    int row;             // the row this thread stores
    int trow;            // that row within the tile
    int b;               // batch
    int lane;
    uint32_t tempty;     // barrier to hand the accumulator back on (cluster address)
    int contrib_first, contrib_count, cs, rank;   // stream-K finisher only
};

// TMEM -> registers -> (stream-K partials) -> alpha * acc + beta * C_in -> bf16/fp32
// -> 128-byte-swizzled shared rows -> TMA store, in 128-byte-wide column chunks,
// double-buffered per warp. Specialised on the output type and on whether
// partials are added, so whole tiles run the lean loop. Returns false when a
// wait ran out (the CTA is aborting).
//
// Partial slots hold [row quarter][column / 4][32 rows][4] floats, so one warp's
// share of a run of columns is contiguous: a finisher copies each contributor's
// share of as many chunks as fit in its staging region in one bulk copy, and
// reads it back conflict-free (lanes on consecutive 16-byte words).
template <int BN, int G, bool OUT_F32, bool FIXUP>
__device__ __forceinline__ bool store_tile(const KernelParams& p, const CUtensorMap* tmC, const EpiTile& e,
                                           uint8_t* stage_ptr, uint32_t stage_base, uint32_t& buf,
                                           const FixStage& fs) {
    constexpr int CW = OUT_F32 ? 32 : 64;             // columns per 128-byte store row
    constexpr int chunks = BN / CW;
    constexpr uint32_t CHUNK_BYTES = (CW / 4) * 512;  // one contributor's chunk for one warp
    const bool use_beta = p.beta != 0.0f;
    const int q = e.trow >> 5;
    // Chunks per staged pass (0: the partials do not fit, add them from global memory).
    const int per_pass = FIXUP && e.contrib_count > 0
                             ? (int)(fs.bytes / (CHUNK_BYTES * (uint32_t)e.contrib_count)) : 0;
    int pass_c0 = 0, pass_n = 0;
    for (int c = 0; c < chunks; ++c) {
        const int col0 = e.n0 + c * CW;
        if (FIXUP && per_pass > 0 && c == pass_c0 + pass_n) {
            // Stage the next pass: every contributor's share of chunks [c, c + pass_n).
            pass_c0 = c;
            pass_n = min(per_pass, chunks - c);
            const uint32_t bytes = (uint32_t)pass_n * CHUNK_BYTES;
            fence_proxy_async_smem();                      // this lane's reads of the previous pass
            __syncwarp();                                  // ... by every lane, before it is overwritten
            if (e.lane == 0) {
                mbar_arrive_expect_tx_local(fs.bar, bytes * (uint32_t)e.contrib_count);
                for (int i = 0; i < e.contrib_count; ++i) {
                    const float4* src =
                        reinterpret_cast<const float4*>(
                            p.workspace +
                            ((long long)(e.contrib_first + i) * e.cs + e.rank) * (long long)(BLOCK_M * BN)) +
                        ((long long)q * (BN / 4) + (long long)c * (CW / 4)) * 32;
                    bulk_load_smem(fs.saddr + (uint32_t)i * bytes, src, bytes, fs.bar);
                }
            }
            if (!wait_bounded(fs.bar, *fs.phase, p, fs.abort_flag, ERR_WAIT_FIXUP, (uint32_t)c, -1)) return false;
            *fs.phase ^= 1u;
        }
        float v[CW];
        {
            uint32_t r[32];
            tmem_ld_32cols(e.t_row + c * CW, r);
            if (!OUT_F32) {
                uint32_t r2[32];
                tmem_ld_32cols(e.t_row + c * CW + 32, r2);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) v[(CW - 32) + i] = __uint_as_float(r2[i]);
            } else {
                tmem_ld_wait();
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        }
        if (FIXUP) {
            // Add the other contributors' partials, in cluster order.
            for (int i = 0; i < e.contrib_count; ++i) {
                const float4* src;
                int stride;
                if (per_pass > 0) {
                    src = reinterpret_cast<const float4*>(
                              fs.ptr + ((size_t)i * pass_n + (size_t)(c - pass_c0)) * CHUNK_BYTES) + e.lane;
                    stride = 32;
                } else {
                    src = reinterpret_cast<const float4*>(
                              p.workspace +
                              ((long long)(e.contrib_first + i) * e.cs + e.rank) * (long long)(BLOCK_M * BN)) +
                          ((long long)q * (BN / 4) + (long long)c * (CW / 4)) * 32 + e.lane;
                    stride = 32;
                }
                // A partial is read once: let L2 drop it first.
                uint64_t pol;
                asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
                for (int j = 0; j < CW / 4; ++j) {
                    float4 a;
                    if (per_pass > 0) {
                        a = src[j * stride];                       // staged: shared memory
                    } else {
                        asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                                     : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w) : "l"(src + j * stride), "l"(pol));
                    }
                    v[4 * j] += a.x;
                    v[4 * j + 1] += a.y;
                    v[4 * j + 2] += a.z;
                    v[4 * j + 3] += a.w;
                }
            }
        }
        if (c == chunks - 1) {
            // All of this accumulator is in registers: hand it back.
            tc_fence_before();
            __syncwarp();
            // CTA-scope release for a CTA's own barrier; cluster scope only when the
            // pair's odd CTA hands back to the even one.
            if (e.lane == 0) {
                if (G == 2) mbar_arrive_cluster(e.tempty);
                else        mbar_arrive_local(e.tempty);
            }
        }
        // alpha * acc + beta * C_in, in fp32.
        if (use_beta) {
            const bool row_ok = e.row < p.M;
            if (OUT_F32) {
                const float* src = static_cast<const float*>(p.c_in) + (long long)e.b * p.stride_c +
                                   (long long)e.row * p.ldc + col0;
#pragma unroll
                for (int i = 0; i < CW; ++i) {
                    const float ci = (row_ok && col0 + i < p.N) ? src[i] : 0.0f;
                    v[i] = fmaf(p.alpha, v[i], p.beta * ci);
                }
            } else {
                const uint16_t* src = static_cast<const uint16_t*>(p.c_in) + (long long)e.b * p.stride_c +
                                      (long long)e.row * p.ldc + col0;
                if (row_ok && col0 + CW <= p.N) {
                    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
                    for (int j = 0; j < CW / 8; ++j) {
                        const uint4 q = s4[j];
                        const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float lo = __uint_as_float(ws[h] << 16);
                            const float hi = __uint_as_float(ws[h] & 0xFFFF0000u);
                            v[8 * j + 2 * h] = fmaf(p.alpha, v[8 * j + 2 * h], p.beta * lo);
                            v[8 * j + 2 * h + 1] = fmaf(p.alpha, v[8 * j + 2 * h + 1], p.beta * hi);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
                        const float ci = (row_ok && col0 + i < p.N) ? __uint_as_float((uint32_t)src[i] << 16) : 0.0f;
                        v[i] = fmaf(p.alpha, v[i], p.beta * ci);
                    }
                }
            }
        } else if (p.alpha != 1.0f) {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] *= p.alpha;
        }
        // Pack one 128-byte row per thread.
        uint32_t w[32];
        if (OUT_F32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        }
        // The buffer about to be written was last used two stores ago.
        if (e.lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* rowp = stage_ptr + buf * EPI_BUF_BYTES + e.lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // 128-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ (r % 8).
            uint4* dst = reinterpret_cast<uint4*>(rowp + ((j ^ (e.lane & 7)) << 4));
            *dst = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (e.lane == 0) {
            tma_store_3d(tmC, stage_base + buf * EPI_BUF_BYTES, col0, e.row0, e.b);
            bulk_commit_group();
        }
        buf ^= 1u;
    }
    return true;
}

template <int BN, int G, int BK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
dgc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const KernelParams p) {
    constexpr int BN_CTA = BN / G;                      // B columns held per CTA
    constexpr uint32_t A_BYTES = BLOCK_M * BK * 2;
    constexpr uint32_t B_BYTES = BN_CTA * BK * 2;
    static_assert(BK == 64 || BK == 128, "a stage is one or two 128-byte swizzle atoms deep");
    constexpr uint32_t TMEM_COLS = 2 * BN;              // two accumulators
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
    static_assert(BN_CTA % 64 == 0, "B slab must be whole 64-column boxes");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint8_t* sA = smem;
    uint8_t* sB = sA + S * A_BYTES;
    uint8_t* sEpi = sB + S * B_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + EPI_SMEM_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + S;
    uint64_t* tfull_bar = bars + 2 * S;
    uint64_t* tempty_bar = bars + 2 * S + 2;
    uint64_t* drain_bar = bars + 2 * S + 4;
    uint64_t* fix_bar = bars + 2 * S + 5;               // one per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 9);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* ring = reinterpret_cast<uint8_t*>(((reinterpret_cast<uintptr_t>(tmem_slot + 6)) + 15) & ~uintptr_t(15));
    const uint32_t ring_resp0 = smem_u32(ring);                                // TILE_RING x 16 bytes
    uint64_t* ring_full = reinterpret_cast<uint64_t*>(ring + 16 * TILE_RING);
    uint64_t* ring_empty = ring_full + TILE_RING;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cx = p.cx, cy = p.cy;
    const int rx = (int)rank % cx;
    const int ry = (int)rank / cx;
    const uint32_t leader = (G == 2) ? (rank & ~1u) : rank;

    // Sharing groups of this CTA.
    const int gA = p.mcast_a ? cy : 1;
    const int idxA = p.mcast_a ? ry : 0;
    const uint32_t maskA = p.mcast_a ? row_mask(rx, cx, cy) : (1u << rank);
    const int gB = p.mcast_b ? cx / G : 1;
    const int idxB = p.mcast_b ? rx / G : 0;
    const uint32_t maskB = p.mcast_b ? col_mask<G>(rx, ry, cx) : (1u << rank);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), (uint32_t)(G * (gA + gB)));
            mbar_init(smem_u32(&empty_bar[s]), (uint32_t)(gA + gB - 1));
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull_bar[i]), 1);
            mbar_init(smem_u32(&tempty_bar[i]), (uint32_t)(G * EPI_WARPS));
        }
        mbar_init(smem_u32(drain_bar), 1);
        for (int i = 0; i < EPI_WARPS; ++i) mbar_init(smem_u32(&fix_bar[i]), 1);
        for (int i = 0; i < TILE_RING; ++i) {
            mbar_init(smem_u32(&ring_full[i]), 1);
            // every CTA's two producers, MMA thread and four epilogue warps read each response
            mbar_init(smem_u32(&ring_empty[i]), (uint32_t)(7 * cx * cy));
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<G>(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish<G>();
    }
    if (warp == 6 && lane == 0) {
        // Fetch the descriptors while thread 0 initialises the barriers, so the first
        // loads do not wait for them after the cluster barrier.
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmC);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Programmatic dependent launch: let the next grid in the stream be scheduled,
    // and touch no global memory (operands, C, workspace, flags, status) before the
    // previous grid has completed and its writes are visible. Both are no-ops for a
    // launch without the attribute.
    const long long cluster = cluster_id_x();
    const long long clusters = num_clusters_x();
    // The producers' operand plans (A: warp 0, B: warp 6).
    auto operand_plan = [&](bool is_a) -> OperandPlan {
        return is_a ? OperandPlan{&tmA, smem_u32(sA), A_BYTES, BLOCK_M, p.a_mn_major, p.a_kmap4, idxA, gA, maskA,
                                  p.a_shared}
                    : OperandPlan{&tmB, smem_u32(sB), B_BYTES, BN_CTA, p.b_mn_major, p.b_kmap4, idxB, gB, maskB,
                                  p.b_shared};
    };
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.prefetch_kb > 0 && (warp == 0 || warp == 6) && lane == 0)
        prefetch_first_stages<G, BK>(p, operand_plan(warp == 0), warp == 0, cx, cy, rx, ry, BN, BN_CTA, cluster,
                                     clusters, p.prefetch_kb);
    // Clock probe: SM cycles and wall nanoseconds from here to the A producer's last
    // load, read by that producer thread where the reads cost nothing: before the wait
    // for the previous grid and after its last load (the clock is the SM's, whatever
    // runs on it; the adds then overlap the last MMAs and the epilogue).
    long long probe_c0 = 0;
    uint64_t probe_t0 = 0;
    if (p.clk && threadIdx.x == 0) {
        probe_c0 = clock64();
        probe_t0 = globaltimer_ns();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    ClcCtx clc_ctx;
    clc_ctx.resp0 = ring_resp0;
    clc_ctx.full0 = smem_u32(&ring_full[0]);
    clc_ctx.empty_rank0 = mapa(smem_u32(&ring_empty[0]), 0);
    clc_ctx.cs = (uint32_t)(cx * cy);
    clc_ctx.abort_flag = abort_flag;
    clc_ctx.consumed = 0;
    clc_ctx.arrive = true;

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------------------ producers (A: warp 0, B: warp 6)
        if (lane == 0) {
            const bool is_a = warp == 0;
            const OperandPlan op = operand_plan(is_a);
            prefetch_tmap(op.tmap);
            if (p.a_l2 != L2_HINT_NONE)
                produce<G, BK, WALK_ONE_WIDE>(p, op, is_a, smem_u32(&full_bar[0]), smem_u32(&empty_bar[0]), rank,
                                              leader, cx, cy, rx, ry, BN, BN_CTA, abort_flag, cluster, clusters, S,
                                              &clc_ctx, smem_u32(&ring_empty[0]));
            else if (p.k_serpentine)
                produce<G, BK, WALK_SERPENTINE>(p, op, is_a, smem_u32(&full_bar[0]), smem_u32(&empty_bar[0]), rank,
                                                leader, cx, cy, rx, ry, BN, BN_CTA, abort_flag, cluster, clusters, S,
                                                &clc_ctx, smem_u32(&ring_empty[0]));
            else
                produce<G, BK, WALK_PLAIN>(p, op, is_a, smem_u32(&full_bar[0]), smem_u32(&empty_bar[0]), rank,
                                           leader, cx, cy, rx, ry, BN, BN_CTA, abort_flag, cluster, clusters, S,
                                           &clc_ctx, smem_u32(&ring_empty[0]));
            if (p.clk && is_a) {
                // One slot of three counters per SM: no two co-resident CTAs add to the same word.
                unsigned long long* slot = p.clk + 3 * (smid() % CLOCK_PROBE_SLOTS);
                atomicAdd(&slot[0], (unsigned long long)(clock64() - probe_c0));
                atomicAdd(&slot[1], (unsigned long long)(globaltimer_ns() - probe_t0));
                atomicAdd(&slot[2], 1ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == leader) {
            constexpr uint32_t UMMA_M = BLOCK_M * G;
            const uint32_t idesc = instr_desc_bf16(UMMA_M, BN, p.a_mn_major != 0, p.b_mn_major != 0);
            // Everyone who writes into this pair's shared memory gets the release.
            uint32_t empty_mask = maskA | maskB;
            if (G == 2) {
                const int px = rx ^ 1;
                const uint32_t pr = (uint32_t)(px + cx * ry);
                empty_mask |= (p.mcast_a ? row_mask(px, cx, cy) : (1u << pr)) |
                              (p.mcast_b ? col_mask<G>(px, ry, cx) : (1u << pr));
            }
            const bool local_only = (empty_mask == (1u << rank));
            // Descriptors advance by adding (byte offset >> 4) to the start-address
            // field (shared addresses stay below 256 KB, so the field cannot carry).
            // K step k (16 elements): MN-major -> 16 K rows further (k * 2048 B);
            // K-major -> atom k/4 (rows * 128 B apart), 32 B into the row per step.
            uint32_t a_koff[BK / 16], b_koff[BK / 16];
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                a_koff[k] = p.a_mn_major ? (uint32_t)(k * 2048) >> 4
                                         : (uint32_t)((k >> 2) * BLOCK_M * 128 + (k & 3) * 32) >> 4;
                b_koff[k] = p.b_mn_major ? (uint32_t)(k * 2048) >> 4
                                         : (uint32_t)((k >> 2) * BN_CTA * 128 + (k & 3) * 32) >> 4;
            }
            const uint64_t adesc0 = smem_desc_sw128(smem_u32(sA), p.a_mn_major != 0, BK * 128);
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sB), p.b_mn_major != 0, BK * 128);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t local_tile = 0;
            bool ok = true;
            WorkIter wi;
            wi.init(p, cluster, clusters, &clc_ctx);
            Work w;
            for (; ok && wi.next(p, w); ++local_tile) {
                const long long t = w.tile;
                const uint32_t acc = local_tile & 1u;
                const uint32_t acc_phase = (local_tile >> 1) & 1u;
                if (!wait_bounded<G == 2>(smem_u32(&tempty_bar[acc]), acc_phase ^ 1u, p, abort_flag,
                                          ERR_WAIT_TMEM_EMPTY, acc, t)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {     // stages arrive in the producers' k order
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase, p, abort_flag,
                                      ERR_WAIT_FULL, (uint32_t)stage, t)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t a_st = adesc0 + ((stage * A_BYTES) >> 4);
                    const uint64_t b_st = bdesc0 + ((stage * B_BYTES) >> 4);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16<G>(d_tmem, a_st + a_koff[k], b_st + b_koff[k], idesc,
                                    (kb > w.kb0 || k > 0) ? 1u : 0u);
                    const uint32_t eb = smem_u32(&empty_bar[stage]);
                    if (local_only) mma_commit<G>(eb);
                    else            mma_commit_mcast<G>(eb, (uint16_t)empty_mask);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                const uint32_t fb = smem_u32(&tfull_bar[acc]);
                if (G == 1) mma_commit<G>(fb);
                else        mma_commit_mcast<G>(fb, (uint16_t)(3u << leader));
            }
            if (*abort_flag) {
                // Let issued MMAs finish before the accumulators are freed.
                mma_commit<G>(smem_u32(drain_bar));
                wait_bounded(smem_u32(drain_bar), 0, p, abort_flag, ERR_WAIT_DRAIN, 0, -1);
            }
        } else if (lane == 0 && p.clc) {
            // The pair's odd CTA issues no MMA but still reads every tile id.
            WorkIter wi;
            wi.init(p, cluster, clusters, &clc_ctx);
            Work w;
            while (wi.next(p, w)) {
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                           // TMEM lane quadrant of this warp
        const int ew = warp - 2;                          // staging buffers of this warp
        const uint32_t stage_base = smem_u32(sEpi + ew * 2 * EPI_BUF_BYTES);
        uint8_t* stage_ptr = sEpi + ew * 2 * EPI_BUF_BYTES;
        const int cs = cx * cy;
        const long long slot = cluster * cs + rank;       // this CTA's stream-K workspace slot
        uint32_t local_tile = 0;
        uint32_t buf = 0;
        // Where this warp hands accumulators back: the pair's even CTA for the pair MMA.
        const uint32_t tempty_addr = (G == 2) ? mapa(smem_u32(&tempty_bar[0]), leader) : smem_u32(&tempty_bar[0]);
        ClcCtx epi_clc = clc_ctx;
        epi_clc.arrive = lane == 0;
        uint32_t fix_phase = 0;
        const uint32_t ring_bytes = (uint32_t)S * (A_BYTES + B_BYTES);
        const uint32_t region = (ring_bytes / EPI_WARPS) & ~511u;
        const FixStage fs{sA + ew * region, smem_u32(sA) + (uint32_t)ew * region, region, smem_u32(&fix_bar[ew]),
                          &fix_phase, abort_flag};
        WorkIter wi;
        wi.init(p, cluster, clusters, &epi_clc);
        Work w;
        // A warp whose wait fails goes on walking the (deterministic) work list
        // without doing the work, so it still joins every named barrier the
        // other epilogue warps reach: none is ever left waiting there alone.
        bool dead = false;
        for (;; ++local_tile) {
            if (!wi.next(p, w)) break;
            const long long t = w.tile;
            const uint32_t acc = local_tile & 1u;
            const uint32_t acc_phase = (local_tile >> 1) & 1u;
            if (!dead && !wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, p, abort_flag,
                                       ERR_WAIT_TMEM_FULL, acc, t))
                dead = true;
            if (dead) {
                // the named barriers the live warps reach for this work
                if (w.kind == WORK_PARTIAL) epilogue_bar();
                if (w.kind == WORK_FINISHER) { epilogue_bar(); epilogue_bar(); }
                continue;
            }
            tc_fence_after();
            const TileCoord tc = tile_coord(p, t);
            const int m0 = (tc.ctm * cx + rx) * BLOCK_M;
            const int n0 = (tc.ctn * cy + ry) * BN;
            const int trow = q * 32 + lane;               // row of the tile this thread owns
            const int row = m0 + trow;                    // global row this thread stores
            const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            if (w.kind == WORK_PARTIAL) {
                // Part of a tile another cluster finishes: park the fp32 partial. A slot
                // holds [row quarter][column / 4][32 rows][4] floats: the 32 rows of a
                // warp write 512 contiguous bytes per store, and the warp's share of the
                // slot is contiguous for the finisher's bulk copies.
                float4* dst = reinterpret_cast<float4*>(p.workspace + slot * (long long)(BLOCK_M * BN)) +
                              (long long)q * (BN / 4) * 32 + lane;
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32cols(t_row + c * 32, r);
                    tmem_ld_wait();
                    if (c == BN / 32 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (G == 2) mbar_arrive_cluster(tempty_addr + 8u * acc);
                            else        mbar_arrive_local(tempty_addr + 8u * acc);
                        }
                    }
                    // Kept in L2 at high priority: the finisher reads the partial back
                    // only after this cluster's whole tiles have streamed their operands.
                    uint64_t pol;
                    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;"
                                     :: "l"(dst + (c * 8 + j) * 32), "f"(__uint_as_float(r[4 * j])),
                                        "f"(__uint_as_float(r[4 * j + 1])), "f"(__uint_as_float(r[4 * j + 2])),
                                        "f"(__uint_as_float(r[4 * j + 3])), "l"(pol) : "memory");
                }
                __threadfence();
                epilogue_bar();
                if (warp == 2 && lane == 0) st_release_gpu(&p.flags[slot], 1u);
                continue;
            }
            if (w.kind == WORK_FINISHER) {
                // Wait until every later contributor of this tile has parked its partial.
                if (warp == 2 && lane == 0) {
                    for (int i = 0; i < w.contrib_count; ++i) {
                        const unsigned int* f = &p.flags[(long long)(w.contrib_first + i) * cs + rank];
                        const uint64_t c0 = clock_cycles();
                        while (ld_acquire_gpu(f) != 1u) {
                            if (*abort_flag) break;
                            if (clock_cycles() - c0 > 2ull * p.timeout_ns) {
                                report_timeout(p, ERR_WAIT_PARTIAL, (uint32_t)(w.contrib_first + i), t);
                                *abort_flag = 1;
                                break;
                            }
                        }
                    }
                }
                epilogue_bar();
            }
            const EpiTile et{t_row, n0, m0 + q * 32, row, trow, tc.b, lane, tempty_addr + 8u * acc,
                             w.contrib_first, w.contrib_count, cs, (int)rank};
            FixStage fsw = fs;
            if (!w.last) fsw.bytes = 0;                   // loads still land in the ring
            bool stored;
            if (p.out_f32) {
                if (w.kind == WORK_FINISHER) stored = store_tile<BN, G, true, true>(p, &tmC, et, stage_ptr, stage_base, buf, fsw);
                else                         stored = store_tile<BN, G, true, false>(p, &tmC, et, stage_ptr, stage_base, buf, fsw);
            } else {
                if (w.kind == WORK_FINISHER) stored = store_tile<BN, G, false, true>(p, &tmC, et, stage_ptr, stage_base, buf, fsw);
                else                         stored = store_tile<BN, G, false, false>(p, &tmC, et, stage_ptr, stage_base, buf, fsw);
            }
            if (!stored) dead = true;
            if (w.kind == WORK_FINISHER) {
                // All four warps have read the partials: lower the contributors' flags
                // for the next launch (which starts after this one in stream order).
                epilogue_bar();
                if (warp == 2 && lane == 0)
                    for (int i = 0; i < w.contrib_count; ++i)
                        p.flags[(long long)(w.contrib_first + i) * cs + rank] = 0u;
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (*abort_flag) {
        // Give any copy still in flight time to land before the CTA exits.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000ull) { }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<G>(tmem_base, TMEM_COLS);
    }
}

}  // namespace dgc
