// Fused attention forward for sm_103a (see include/attention.h).
//
// "Hopper TMA Multicast 深度解析与实测", section 经典应用场景: the CTAs of a
// cluster hold adjacent query tiles of the same (batch, head) and need the
// same K and V tiles, so each K/V tile is fetched once and multicast to all
// of them, every issuer arming each receiver's mbarrier (through mapa) before
// it issues (section 深度机制剖析).
//
// One CTA = two 128-row query tiles (Q0, Q1) of one (batch, head). Tensor
// memory holds both score tiles and both output accumulators (4 x 128 of its
// 512 columns); the probabilities P_i overwrite the first 64 columns of S_i
// as packed bf16 and feed O_i += P_i V_j straight from tensor memory, so no
// score or probability ever touches shared memory.
//
// Roles (384 threads):
//   warp 0      producer: Q0 and Q1 once, then K_0, V_0, K_1, V_1, ... into a
//               ring of four 32 KB slots (this CTA's slice of each, multicast)
//   warp 1      TMEM allocation and MMA issue, per key tile j in the order
//               O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T
//               so the tensor core works on one tile while the other tile's
//               softmax runs (the two softmaxes take turns on the exp unit)
//   warps 2, 3  idle
//   warps 4-7   softmax of tile 0, warps 8-11 softmax of tile 1: one query row
//               per thread, online softmax in base 2 with a reference max that
//               moves (rescaling O in TMEM) only when the row max grows by
//               more than 2^8; at the end O / l and the log-sum-exp.
//
// Pair mode ("Clusters, distributed shared memory & cluster launch control",
// section "Two CTAs, one MMA"): a 2-CTA cluster issues tcgen05.mma.cta_group::2
// from its even CTA. S_i = Q_i K_j^T runs as one M = 256 MMA over both CTAs'
// Q_i (each CTA's scores land in its own TMEM), each CTA holding half of every
// K tile (64 keys) and half of every V tile (64 of the d columns), so per SM
// the score MMA reads 6 KB of shared memory per K step instead of 8 and P V
// 2 KB instead of 4. The odd CTA's softmax warps hand P back to the even CTA's
// barrier; completions are multicast to both CTAs.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "attention.h"
#include "densegemm.h"
#include "host_env.h"
#include "ptx.cuh"

namespace {

using namespace dgc;

constexpr int TQ = 128;                  // queries per tile
constexpr int QT = 2;                    // query tiles per CTA
constexpr int TK = 128;                  // keys per tile
constexpr int THREADS = 384;
constexpr uint32_t ATOM_BYTES = 128 * 128;      // one 64-element swizzle atom of a 128-row tile
constexpr int NS = 4;                           // ring slots; K and V tiles alternate
constexpr float RESCALE_THRESHOLD = 8.0f;       // log2 units: move the reference max past 2^8 growth
// A Q, K or V tile is 128 rows of the head dimension (32 KB at 128, 16 KB at 64).
__host__ __device__ constexpr uint32_t tile_bytes(int hd) { return 128u * (uint32_t)hd * 2u; }
constexpr size_t smem_bytes(int hd) { return 1024 + (QT + NS) * (size_t)tile_bytes(hd) + 24 * 8 + 16; }

__device__ unsigned int g_attn_status[4];

struct AttnParams {
    int batch, sq, sk;
    int n_kv;                    // key tiles
    int cluster;
    float scale_log2;            // scale * log2(e)
    int out_f32;
    void* out;
    float* lse;
    unsigned long long timeout_ns;
};

__device__ bool attn_wait(uint32_t bar, uint32_t parity, const AttnParams& p, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t c0 = clock_cycles();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (clock_cycles() - c0 > 2ull * p.timeout_ns) {
            if (atomicCAS(&g_attn_status[0], 0u, code) == 0u) {
                g_attn_status[1] = blockIdx.x;
                g_attn_status[2] = blockIdx.z * gridDim.y + blockIdx.y;
                __threadfence();
            }
            return false;
        }
    }
}

// The same wait with a cluster-scope acquire: for barriers a peer CTA arrives on
// with a release (the pair's odd CTA handing its P to the even CTA).
__device__ bool attn_wait_cluster(uint32_t bar, uint32_t parity, const AttnParams& p, uint32_t code) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t c0 = clock_cycles();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (clock_cycles() - c0 > 2ull * p.timeout_ns) {
            if (atomicCAS(&g_attn_status[0], 0u, code) == 0u) {
                g_attn_status[1] = blockIdx.x;
                g_attn_status[2] = blockIdx.z * gridDim.y + blockIdx.y;
                __threadfence();
            }
            return false;
        }
    }
}

// O (+)= P V as one pair MMA: P (packed bf16) from TMEM of both CTAs of the pair.
__device__ __forceinline__ void mma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// K-major 128-row tile as an MMA operand: atoms of 64 elements are 16 KB apart.
__device__ __forceinline__ uint32_t kmajor_koff(int k) { return (uint32_t)((k >> 2) * ATOM_BYTES + (k & 3) * 32) >> 4; }
// Half a K tile (64 keys) in pair mode: atoms 8 KB apart.
__device__ __forceinline__ uint32_t kmajor_koff_half(int k) {
    return (uint32_t)((k >> 2) * (ATOM_BYTES / 2) + (k & 3) * 32) >> 4;
}
// MN-major tile (V: 128 keys x 128 d): K step of 16 keys = 16 rows of 128 bytes.
__device__ __forceinline__ uint32_t mnmajor_koff(int k) { return (uint32_t)(k * 2048) >> 4; }

template <bool PAIR, bool CAUSAL, int HD>
__global__ void __launch_bounds__(THREADS, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    // Ring: NS slots of a whole K or V tile, or (pair) twice as many of half tiles.
    constexpr int NSL = PAIR ? 2 * NS : NS;
    static_assert(HD == 64 || HD == 128, "head dimension 64 or 128");
    static_assert(!PAIR || HD == 128, "the pair MMA splits 128 head columns");
    constexpr uint32_t TILE_BYTES = tile_bytes(HD);
    constexpr int ATOMS = HD / 64;                    // 128-byte swizzle atoms across a Q or K row
    constexpr uint32_t SLOT_BYTES = PAIR ? TILE_BYTES / 2 : TILE_BYTES;
    constexpr int G = PAIR ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                                   // QT tiles
    uint8_t* ring = sQ + QT * TILE_BYTES;                 // NS slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + NS * TILE_BYTES);
    uint64_t* q_full = bars;                 // 1
    uint64_t* kv_full = bars + 1;            // NSL
    uint64_t* kv_empty = bars + 1 + NSL;     // NSL
    uint64_t* s_full = bars + 1 + 2 * NSL;   // QT: S_i written
    uint64_t* p_full = s_full + QT;          // QT: P_i written (and O_i rescaled)
    uint64_t* pv_done = p_full + QT;         // QT: O_i += P_i V_j completed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pv_done + QT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = p.cluster;
    const uint32_t rank = c > 1 ? cluster_ctarank() : 0u;
    const uint16_t all = (uint16_t)((1u << c) - 1u);
    // Not causal: grid x = query blocks, heads in grid y, continued in grid z past
    // 65535. Causal: grid x = heads x the c blocks of a cluster, grid y = groups of c
    // query blocks, last group first, so every head's longest rows start before any
    // shorter ones. A cluster spans grid x within one head either way, so it leaves
    // together when the grid runs past the batch.
    int b, qblk, cluster_last_qblk;
    if (CAUSAL) {
        b = (int)(blockIdx.x / (unsigned)c + blockIdx.z * (gridDim.x / (unsigned)c));
        const int group = (int)gridDim.y - 1 - (int)blockIdx.y;
        qblk = group * c + (int)(blockIdx.x % (unsigned)c);
        cluster_last_qblk = group * c + c - 1;
    } else {
        b = (int)(blockIdx.z * gridDim.y + blockIdx.y);
        qblk = (int)blockIdx.x;
        cluster_last_qblk = qblk;
    }
    if (b >= p.batch) return;
    const int q0 = qblk * (QT * TQ);
    int n_kv = p.n_kv;
    if (CAUSAL) {
        // A cluster's CTAs share every K/V tile: walk the key tiles its last query needs;
        // rows before the diagonal see the later keys masked.
        const long long last_q = min((long long)p.sq, (long long)(cluster_last_qblk + 1) * (QT * TQ)) - 1;
        const long long keys = min((long long)p.sk, last_q + 1);
        n_kv = (int)((keys + TK - 1) / TK);
    }
    // Key tiles each query tile of this CTA scores: the cluster's count, or (causal,
    // single-CTA MMAs) only those up to the tile's last query. Past its count a tile
    // issues no MMA, but the last tile still releases every K/V slot.
    auto n_kv_tile = [&](int i) -> int {
        if (!CAUSAL || PAIR) return n_kv;
        const long long keys = min((long long)p.sk, (long long)q0 + (i + 1) * TQ);
        return max(1, min(n_kv, (int)((keys + TK - 1) / TK)));
    };

    if (threadIdx.x == 0) {
        // Pair: the even CTA's q_full and kv_full count both CTAs' arms and bytes, its
        // p_full both CTAs' softmax warps; every release and completion is multicast.
        mbar_init(smem_u32(q_full), PAIR ? 2u : 1u);
        for (int s = 0; s < NSL; ++s) {
            mbar_init(smem_u32(&kv_full[s]), PAIR ? 2u : (uint32_t)c);    // one arm per issuer of a slice
            mbar_init(smem_u32(&kv_empty[s]), PAIR ? 1u : (uint32_t)c);   // one release per consumer CTA
        }
        for (int i = 0; i < QT; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&p_full[i]), PAIR ? 8u : 4u);
            mbar_init(smem_u32(&pv_done[i]), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<G>(smem_u32(tmem_slot), 512);
        tmem_relinquish<G>();
    }
    tc_fence_before();
    __syncthreads();
    if (c > 1) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;        // columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512)

    if (PAIR && warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer (pair)
        // This CTA's Q tiles and its half of each K tile (64 keys) and V tile (64 of the
        // d columns), each arming and signalling the even CTA's barrier.
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        const uint32_t leader = rank & ~1u;
        const int h = (int)(rank & 1u);
        const uint32_t qb = mapa(smem_u32(q_full), leader);
        mbar_arrive_expect_tx_cluster(qb, QT * TILE_BYTES);
        for (int i = 0; i < QT; ++i)
            tma_load_4d_pair(smem_u32(sQ + i * TILE_BYTES), &tmQ, qb, 0, q0 + i * TQ, 0, b);
        const int loads = 2 * n_kv;
        for (int n = 0; n < loads; ++n) {
            const int s = n % NSL;
            const uint32_t ph = (uint32_t)(n / NSL) & 1u;
            if (!attn_wait(smem_u32(&kv_empty[s]), ph ^ 1u, p, 1)) break;
            const uint32_t fb = mapa(smem_u32(&kv_full[s]), leader);
            mbar_arrive_expect_tx_cluster(fb, SLOT_BYTES);
            const uint32_t dst = smem_u32(ring + s * SLOT_BYTES);
            const int key0 = (n >> 1) * TK;
            if ((n & 1) == 0) tma_load_4d_pair(dst, &tmK, fb, 0, key0 + h * (TK / 2), 0, b);
            else              tma_load_3d_pair(dst, &tmV, fb, h * 64, key0, b);
        }
        // Every slot this thread filled is released before exit.
        for (int n = loads; n < loads + NSL; ++n) {
            const int s = n % NSL;
            if (!attn_wait(smem_u32(&kv_empty[s]), ((uint32_t)(n / NSL) & 1u) ^ 1u, p, 1)) break;
        }
    } else if (PAIR && warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer (pair)
        // Only the even CTA issues; the order matches the single-CTA kernel below.
        if ((rank & 1u) == 0) {
            const uint16_t pairm = (uint16_t)(3u << rank);
            const uint32_t idesc_s = instr_desc_bf16(2 * TQ, TK, false, false);
            const uint32_t idesc_o = instr_desc_bf16(2 * TQ, HD, false, true);
            const uint64_t ring_k = smem_desc_sw128(smem_u32(ring), false, 0);
            const uint64_t ring_v = smem_desc_sw128(smem_u32(ring), true, SLOT_BYTES);
            bool ok = attn_wait(smem_u32(q_full), 0, p, 2);
            auto issue_s = [&](int i, int j) -> bool {
                const int n = 2 * j, s = n % NSL;
                if (i == 0) {
                    if (!attn_wait(smem_u32(&kv_full[s]), (uint32_t)(n / NSL) & 1u, p, 3)) return false;
                    tc_fence_after();
                }
                const uint64_t dq = smem_desc_sw128(smem_u32(sQ + i * TILE_BYTES), false, 0);
                const uint64_t dk = ring_k + ((s * SLOT_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    mma_bf16<2>(tmem + i * TK, dq + kmajor_koff(k), dk + kmajor_koff_half(k), idesc_s, k > 0 ? 1u : 0u);
                mma_commit_mcast<2>(smem_u32(&s_full[i]), pairm);
                if (i == QT - 1) mma_commit_mcast<2>(smem_u32(&kv_empty[s]), pairm);
                return true;
            };
            auto issue_pv = [&](int i, int j) -> bool {
                const int n = 2 * j + 1, s = n % NSL;
                if (i == 0 && !attn_wait(smem_u32(&kv_full[s]), (uint32_t)(n / NSL) & 1u, p, 4)) return false;
                if (!attn_wait_cluster(smem_u32(&p_full[i]), (uint32_t)j & 1u, p, 5)) return false;
                tc_fence_after();
                const uint64_t dv = ring_v + ((s * SLOT_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < TK / 16; ++k)
                    mma_bf16_ts_pair(tmem + 2 * TK + i * HD, tmem + i * TK + k * 8, dv + mnmajor_koff(k), idesc_o,
                                     (j > 0 || k > 0) ? 1u : 0u);
                mma_commit_mcast<2>(smem_u32(&pv_done[i]), pairm);
                if (i == QT - 1) mma_commit_mcast<2>(smem_u32(&kv_empty[s]), pairm);
                return true;
            };
            if (ok) ok = issue_s(0, 0) && issue_s(1, 0);
            for (int j = 0; ok && j < n_kv; ++j) {
                const bool more = j + 1 < n_kv;
                ok = issue_pv(0, j) && (!more || issue_s(0, j + 1)) && issue_pv(1, j) && (!more || issue_s(1, j + 1));
            }
        }
    } else if (!PAIR && warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_arrive_expect_tx_local(smem_u32(q_full), QT * TILE_BYTES);
        for (int i = 0; i < QT; ++i)
            tma_load_4d(smem_u32(sQ + i * TILE_BYTES), &tmQ, smem_u32(q_full), 0, q0 + i * TQ, 0, b);
        // This CTA's slice of each shared tile. K (K-major, HD / 64 atoms): whole atoms
        // first, then rows within an atom. V (MN-major, HD / 64 boxes of 64 d columns x
        // 128 keys): a band of key rows of every box.
        int k_atom0 = 0, k_r0 = 0;
        if (c <= ATOMS) { k_atom0 = (int)rank * (ATOMS / c); }
        else { k_atom0 = (int)rank / (c / ATOMS); k_r0 = ((int)rank % (c / ATOMS)) * (TK / (c / ATOMS)); }
        const int v_r0 = (int)rank * (TK / c);
        const uint32_t slice_bytes = TILE_BYTES / (uint32_t)c;
        const int loads = 2 * n_kv;
        for (int n = 0; n < loads; ++n) {
            const int s = n % NS;
            const uint32_t ph = (uint32_t)(n / NS) & 1u;
            if (!attn_wait(smem_u32(&kv_empty[s]), ph ^ 1u, p, 1)) break;
            const uint32_t fb = smem_u32(&kv_full[s]);
            for (int r = 0; r < c; ++r) {
                if (r == (int)rank) mbar_arrive_expect_tx_local(fb, slice_bytes);
                else mbar_arrive_expect_tx_cluster(mapa(fb, (uint32_t)r), slice_bytes);
            }
            const uint32_t tile = smem_u32(ring + s * TILE_BYTES);
            const int key0 = (n >> 1) * TK;
            if ((n & 1) == 0) {
                const uint32_t dst = tile + (uint32_t)(k_atom0 * ATOM_BYTES + k_r0 * 128);
                if (c > 1) tma_load_4d_mcast(dst, &tmK, fb, 0, key0 + k_r0, k_atom0, b, all);
                else       tma_load_4d(dst, &tmK, fb, 0, key0, 0, b);
            } else {
                for (int box = 0; box < HD / 64; ++box) {
                    const uint32_t dst = tile + (uint32_t)(box * TK * 128 + v_r0 * 128);
                    if (c > 1) tma_load_3d_mcast(dst, &tmV, fb, box * 64, key0 + v_r0, b, all);
                    else       tma_load_3d(dst, &tmV, fb, box * 64, key0, b);
                }
            }
        }
        // Every slot this thread filled is released by all receivers before exit.
        for (int n = loads; n < loads + NS; ++n) {
            const int s = n % NS;
            if (!attn_wait(smem_u32(&kv_empty[s]), ((uint32_t)(n / NS) & 1u) ^ 1u, p, 1)) break;
        }
    } else if (!PAIR && warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idesc_s = instr_desc_bf16(TQ, TK, false, false);    // Q (K-major) x K^T (K-major)
        const uint32_t idesc_o = instr_desc_bf16(TQ, HD, false, true);     // P (TMEM) x V (MN-major)
        const uint64_t ring_k = smem_desc_sw128(smem_u32(ring), false, 0);
        const uint64_t ring_v = smem_desc_sw128(smem_u32(ring), true, TK * 128);
        bool ok = attn_wait(smem_u32(q_full), 0, p, 2);
        // S_i = Q_i K_j^T; the second tile's commit releases K_j's slot.
        auto issue_s = [&](int i, int j) -> bool {
            const int n = 2 * j, s = n % NS;
            if (i == 0) {
                if (!attn_wait(smem_u32(&kv_full[s]), (uint32_t)(n / NS) & 1u, p, 3)) return false;
                tc_fence_after();
            }
            if (j < n_kv_tile(i)) {
                const uint64_t dq = smem_desc_sw128(smem_u32(sQ + i * TILE_BYTES), false, 0);
                const uint64_t dk = ring_k + ((s * TILE_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    mma_bf16<1>(tmem + i * TK, dq + kmajor_koff(k), dk + kmajor_koff(k), idesc_s, k > 0 ? 1u : 0u);
                mma_commit<1>(smem_u32(&s_full[i]));
            }
            if (i == QT - 1) {
                if (c > 1) mma_commit_mcast<1>(smem_u32(&kv_empty[s]), all);
                else       mma_commit<1>(smem_u32(&kv_empty[s]));
            }
            return true;
        };
        // O_i += P_i V_j with P_i from TMEM; the second tile's commit releases V_j's slot.
        auto issue_pv = [&](int i, int j) -> bool {
            const int n = 2 * j + 1, s = n % NS;
            if (i == 0 && !attn_wait(smem_u32(&kv_full[s]), (uint32_t)(n / NS) & 1u, p, 4)) return false;
            if (j < n_kv_tile(i)) {
                if (!attn_wait(smem_u32(&p_full[i]), (uint32_t)j & 1u, p, 5)) return false;
                tc_fence_after();
                const uint64_t dv = ring_v + ((s * TILE_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < TK / 16; ++k)
                    mma_bf16_ts(tmem + 2 * TK + i * HD, tmem + i * TK + k * 8, dv + mnmajor_koff(k), idesc_o,
                                (j > 0 || k > 0) ? 1u : 0u);
                mma_commit<1>(smem_u32(&pv_done[i]));
            }
            if (i == QT - 1) {
                if (c > 1) mma_commit_mcast<1>(smem_u32(&kv_empty[s]), all);
                else       mma_commit<1>(smem_u32(&kv_empty[s]));
            }
            return true;
        };
        if (ok) ok = issue_s(0, 0) && issue_s(1, 0);
        for (int j = 0; ok && j < n_kv; ++j) {
            const bool more = j + 1 < n_kv;
            ok = issue_pv(0, j) && (!more || issue_s(0, j + 1)) && issue_pv(1, j) && (!more || issue_s(1, j + 1));
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- softmax
        const int ti = (warp - 4) >> 2;              // query tile
        const int qd = warp & 3;                     // TMEM lane quadrant
        const int row = qd * 32 + lane;              // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
        const uint32_t tS = lane_base + ti * TK;
        const uint32_t tO = lane_base + 2 * TK + ti * HD;
        const float cs = p.scale_log2;
        float m_ref = -INFINITY;                     // reference max, base-2 units
        float l = 0.0f;                              // running sum of 2^(x - m_ref)
        bool ok = true;
        const int q_row = q0 + ti * TQ + row;       // this thread's query
        const int n_kv_mine = n_kv_tile(ti);
        for (int j = 0; j < n_kv_mine; ++j) {
            if (!attn_wait(smem_u32(&s_full[ti]), (uint32_t)j & 1u, p, 7)) { ok = false; break; }
            tc_fence_after();
            uint32_t x[TK];
            tmem_ld_128cols_wait(tS, x);
            int valid = p.sk - j * TK;               // keys of this tile inside the sequence
            if (CAUSAL) valid = min(valid, q_row - j * TK + 1);     // and not after this query
            if (valid < TK) {
#pragma unroll
                for (int i = 0; i < TK; ++i)
                    if (i >= valid) x[i] = __float_as_uint(-INFINITY);
            }
            // Row max: eight independent chains of three-input maxima.
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(x[2 * k]), __uint_as_float(x[2 * k + 1]));
#pragma unroll
            for (int i = 16; i < TK; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    m8[k] = max3f(m8[k], __uint_as_float(x[i + 2 * k]), __uint_as_float(x[i + 2 * k + 1]));
            const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
            const float m_new = mx * cs;
            float alpha = 1.0f;                      // factor for O and l when the reference moves
            if (j == 0) {
                m_ref = m_new;
            } else if (m_new > m_ref + RESCALE_THRESHOLD) {
                alpha = ex2_approx(m_ref - m_new);
                m_ref = m_new;
            }
            // P over the first 64 columns of S: keys 2c and 2c+1 packed in column c.
            // Pairs of keys go through packed fp32 arithmetic: x * scale - m_ref in one
            // fma.f32x2, the row sum in two f32x2 accumulators.
            const uint64_t cs2 = f32x2(cs, cs);
            const uint64_t neg2 = f32x2(-m_ref, -m_ref);
            uint64_t ls2[2] = {f32x2(0.0f, 0.0f), f32x2(0.0f, 0.0f)};
#pragma unroll
            for (int h = 0; h < TK / 32; ++h) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t t = fma_f32x2(
                        f32x2(__uint_as_float(x[32 * h + 2 * i]), __uint_as_float(x[32 * h + 2 * i + 1])), cs2, neg2);
                    float t0, t1;
                    f32x2_split(t, t0, t1);
                    const float p0 = ex2_approx(t0);
                    const float p1 = ex2_approx(t1);
                    ls2[i & 1] = add_f32x2(ls2[i & 1], f32x2(p0, p1));
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st_16cols(tS + h * 16, pk);
            }
            {
                float a0, a1, b0, b1;
                f32x2_split(ls2[0], a0, a1);
                f32x2_split(ls2[1], b0, b1);
                l = fmaf(l, alpha, (a0 + a1) + (b0 + b1));
            }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                // O_i is stable once P_i V_{j-1} has completed.
                if (!attn_wait(smem_u32(&pv_done[ti]), (uint32_t)(j - 1) & 1u, p, 8)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int h = 0; h < HD / 32; ++h) {
                    uint32_t r[32];
                    tmem_ld_32cols_wait(tO + h * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    tmem_st_32cols(tO + h * 32, r);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // The pair's odd CTA hands its P to the even CTA's barrier with a
                // cluster-scope release (the even CTA's MMAs read this CTA's TMEM).
                if (!PAIR || (rank & 1u) == 0) mbar_arrive_local(smem_u32(&p_full[ti]));
                else                           mbar_arrive_cluster(mapa(smem_u32(&p_full[ti]), rank & ~1u));
            }
        }
        // Final normalisation: O / l, and lse = (m_ref + log2 l) * ln 2.
        if (ok && attn_wait(smem_u32(&pv_done[ti]), (uint32_t)(n_kv_mine - 1) & 1u, p, 9)) {
            tc_fence_after();
            const int q = q0 + ti * TQ + row;
            const float inv = 1.0f / l;
            for (int h = 0; h < HD / 32; ++h) {
                uint32_t r[32];
                tmem_ld_32cols_wait(tO + h * 32, r);
                if (q < p.sq) {
                    const long long off = ((long long)b * p.sq + q) * HD + h * 32;
                    if (p.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + off);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                                 __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + off);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * i]) * inv, __uint_as_float(r[8 * i + 1]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv));
                    }
                }
            }
            if (p.lse && q < p.sq) p.lse[(long long)b * p.sq + q] = (m_ref + log2f(l)) * 0.69314718055994531f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (c > 1) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<G>(tmem, 512);
    }
}

thread_local char g_attn_err[256];

gemm_status_t afail(gemm_status_t s, const char* m) {
    snprintf(g_attn_err, sizeof g_attn_err, "%s", m);
    return s;
}

PFN_cuTensorMapEncodeTiled_v12000 attn_encoder() {
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

bool encode(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" gemm_status_t attention_forward_run(const void* Q, const void* K, const void* V, void* O, float* lse,
                                               int64_t batch, int64_t sq, int64_t sk, int64_t d, float scale,
                                               int out_f32, int cluster, int cta_group, int causal,
                                               void* stream) {
    if (batch < 0 || sq < 0 || sk < 0) return afail(GEMM_ERR_INVALID_ARG, "negative size");
    if (batch == 0 || sq == 0) return GEMM_OK;
    if (sk == 0) return afail(GEMM_ERR_INVALID_ARG, "sk must be at least 1");
    if (d != 64 && d != 128) return afail(GEMM_ERR_UNSUPPORTED, "head dimension must be 64 or 128");
    if (cluster != 1 && cluster != 2 && cluster != 4) return afail(GEMM_ERR_UNSUPPORTED, "cluster must be 1, 2 or 4");
    if (cta_group != 1 && cta_group != 2) return afail(GEMM_ERR_UNSUPPORTED, "cta_group must be 1 or 2");
    if (cta_group == 2 && cluster != 2) return afail(GEMM_ERR_UNSUPPORTED, "the pair MMA runs in clusters of 2");
    if (cta_group == 2 && d != 128) return afail(GEMM_ERR_UNSUPPORTED, "the pair MMA needs head dimension 128");
    const bool pair = cta_group == 2;
    // Clusters of 2 or 4 single-CTA MMAs multicast every K/V tile: single-GPU only.
    if (cluster > 1 && !pair && dgc_host::world_is_multi_gpu())
        return afail(GEMM_ERR_UNSUPPORTED,
                     "K/V cluster multicast is single-GPU only; WORLD_SIZE > 1 requires cluster 1 or the pair MMA");
    if (!Q || !K || !V || !O) return afail(GEMM_ERR_INVALID_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
         reinterpret_cast<uintptr_t>(O) | reinterpret_cast<uintptr_t>(lse)) & 15u)
        return afail(GEMM_ERR_ALIGNMENT, "Q, K, V, O and lse must be 16-byte aligned");
    if (batch >= (1ll << 31) || sq >= (1ll << 31) || sk >= (1ll << 31)) return afail(GEMM_ERR_INVALID_ARG, "too large");
    auto enc = attn_encoder();
    if (!enc) return afail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap tq, tk, tv;
    const int64_t HD = d;
    const int atoms = (int)(d / 64);                      // 128-byte swizzle atoms across a row
    // Q and K: the k-split view {64, rows, atoms, batch} (atoms 128 bytes apart).
    const cuuint64_t qd[4] = {64, (cuuint64_t)sq, (cuuint64_t)atoms, (cuuint64_t)batch};
    const cuuint64_t qs[3] = {(cuuint64_t)(HD * 2), 128, (cuuint64_t)(sq * HD * 2)};
    const cuuint32_t qb[4] = {64, TQ, (cuuint32_t)atoms, 1};
    const cuuint64_t kd[4] = {64, (cuuint64_t)sk, (cuuint64_t)atoms, (cuuint64_t)batch};
    const cuuint64_t ks[3] = {(cuuint64_t)(HD * 2), 128, (cuuint64_t)(sk * HD * 2)};
    // A K slice: whole atoms first, then bands of rows within an atom; pair mode: half
    // the keys, every atom.
    const int k_rows = pair ? TK / 2 : (cluster <= atoms ? TK : TK / (cluster / atoms));
    const int k_atoms = pair ? atoms : (cluster <= atoms ? atoms / cluster : 1);
    const cuuint32_t kb[4] = {64, (cuuint32_t)k_rows, (cuuint32_t)k_atoms, 1};
    // V: MN-major boxes of 64 d columns x (128 / cluster) keys (pair mode: all 128 keys).
    const cuuint64_t vd[3] = {(cuuint64_t)HD, (cuuint64_t)sk, (cuuint64_t)batch};
    const cuuint64_t vs[2] = {(cuuint64_t)(HD * 2), (cuuint64_t)(sk * HD * 2)};
    const cuuint32_t vb[3] = {64, (cuuint32_t)(pair ? TK : TK / cluster), 1};
    if (!encode(enc, &tq, Q, 4, qd, qs, qb) || !encode(enc, &tk, K, 4, kd, ks, kb) || !encode(enc, &tv, V, 3, vd, vs, vb))
        return afail(GEMM_ERR_INVALID_ARG, "tensor map encode failed");
    AttnParams p;
    memset(&p, 0, sizeof p);
    p.batch = (int)batch;
    p.sq = (int)sq;
    p.sk = (int)sk;
    p.n_kv = (int)((sk + TK - 1) / TK);
    p.cluster = cluster;
    p.scale_log2 = (scale > 0.0f ? scale : 1.0f / sqrtf((float)d)) * 1.4426950408889634f;
    p.out_f32 = out_f32 ? 1 : 0;
    p.out = O;
    p.lse = lse;
    p.timeout_ns = 2000000000ull;
    void* fn;
    if (pair) fn = causal ? reinterpret_cast<void*>(&attention_fwd_kernel<true, true, 128>)
                          : reinterpret_cast<void*>(&attention_fwd_kernel<true, false, 128>);
    else if (d == 128) fn = causal ? reinterpret_cast<void*>(&attention_fwd_kernel<false, true, 128>)
                                   : reinterpret_cast<void*>(&attention_fwd_kernel<false, false, 128>);
    else fn = causal ? reinterpret_cast<void*>(&attention_fwd_kernel<false, true, 64>)
                     : reinterpret_cast<void*>(&attention_fwd_kernel<false, false, 64>);
    const size_t smem = smem_bytes((int)d);
    // Set the shared-memory limit once per device and kernel, so that a steady-state
    // call is one launch (and can be captured into a CUDA graph).
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    static std::atomic<unsigned char> smem_set[64][8];
    std::atomic<unsigned char>& flag = smem_set[dev & 63][(pair ? 1 : 0) + (causal ? 2 : 0) + (d == 64 ? 4 : 0)];
    if (!flag.load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
        flag.store(1, std::memory_order_release);
    }
    long long ctas = (sq + QT * TQ - 1) / (QT * TQ);
    ctas = (ctas + cluster - 1) / cluster * cluster;      // whole clusters; extra CTAs store nothing
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    if (causal && ctas / cluster > 65535)
        return afail(GEMM_ERR_UNSUPPORTED, "causal: at most 65535 groups of query blocks (sq up to 65535 * 256 * cluster)");
    if (causal) {
        const long long hx = batch < (1ll << 30) / cluster ? batch : (1ll << 30) / cluster;
        cfg.gridDim = dim3((unsigned)(hx * cluster), (unsigned)(ctas / cluster), (unsigned)((batch + hx - 1) / hx));
    } else {
        const unsigned gy = (unsigned)(batch < 65535 ? batch : 65535);
        cfg.gridDim = dim3((unsigned)ctas, gy, (unsigned)((batch + gy - 1) / gy));
    }
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&tq, &tk, &tv, &p};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    return GEMM_OK;
}

extern "C" gemm_status_t attention_forward_query_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    unsigned int w[4] = {0, 0, 0, 0};
    e = cudaMemcpyFromSymbol(w, g_attn_status, sizeof w);
    if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    if (w[0] == 0) return GEMM_OK;
    unsigned int z[4] = {0, 0, 0, 0};
    cudaMemcpyToSymbol(g_attn_status, z, sizeof z);
    snprintf(g_attn_err, sizeof g_attn_err, "attention: bounded wait %u expired (q block %u, batch %u)", w[0], w[1], w[2]);
    return GEMM_ERR_DEVICE_TIMEOUT;
}
