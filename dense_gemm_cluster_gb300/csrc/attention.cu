// Fused attention forward for sm_103a (see include/attention.h).
//
// "Hopper TMA Multicast 深度解析与实测", section 经典应用场景: the CTAs of a
// cluster hold adjacent query tiles of the same (batch, head) and need the
// same K and V tiles, so each K/V tile is fetched once and multicast to all
// of them, every issuer arming each receiver's mbarrier (through mapa) before
// it issues (section 深度机制剖析).
//
// One CTA = one 128-row query tile. Roles (224 threads):
//   warp 0      producer: the Q tile once, then K tiles into a 2-stage ring
//   warp 6      producer: V tiles into the same ring
//   warp 1      TMEM allocation and MMA issue: S_j = Q K_j^T into one of two
//               TMEM score buffers, O += P_j V_j into the TMEM output
//   warps 2..5  softmax: one query row per thread; online softmax in base 2
//               with a running reference max that is moved (and O rescaled in
//               TMEM) only when a row's max grows by more than 2^8; P_j goes
//               to shared memory as bf16; finally O / l and the log-sum-exp.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>

#include "attention.h"
#include "densegemm.h"
#include "ptx.cuh"

namespace {

using namespace dgc;

constexpr int TQ = 128;                  // queries per CTA
constexpr int TK = 128;                  // keys per tile
constexpr int HD = 128;                  // head dimension
constexpr int THREADS = 224;
constexpr uint32_t TILE_BYTES = TQ * HD * 2;    // 32 KB: Q, K, V and P tiles alike
constexpr uint32_t ATOM_BYTES = TQ * 128;       // one 64-element swizzle atom of a 128-row tile
constexpr int KV_STAGES = 2;
constexpr float RESCALE_THRESHOLD = 8.0f;       // log2 units: move the reference max past 2^8 growth

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
                g_attn_status[2] = blockIdx.y;
                __threadfence();
            }
            return false;
        }
    }
}

// K-major 128-row tile as an MMA operand: atoms of 64 elements are 16 KB apart.
__device__ __forceinline__ uint32_t kmajor_koff(int k) { return (uint32_t)((k >> 2) * ATOM_BYTES + (k & 3) * 32) >> 4; }
// MN-major tile (V: 128 keys x 128 d): K step of 16 keys = 16 rows of 128 bytes.
__device__ __forceinline__ uint32_t mnmajor_koff(int k) { return (uint32_t)(k * 2048) >> 4; }

__global__ void __launch_bounds__(THREADS, 1)
attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + TILE_BYTES;                       // KV_STAGES tiles
    uint8_t* sV = sK + KV_STAGES * TILE_BYTES;           // KV_STAGES tiles
    uint8_t* sP = sV + KV_STAGES * TILE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + TILE_BYTES);
    uint64_t* q_full = bars;                 // 1
    uint64_t* k_full = bars + 1;             // KV_STAGES
    uint64_t* v_full = bars + 3;             // KV_STAGES
    uint64_t* kv_empty = bars + 5;           // KV_STAGES
    uint64_t* s_full = bars + 7;             // 2
    uint64_t* s_empty = bars + 9;            // 2
    uint64_t* p_full = bars + 11;            // 1
    uint64_t* pv_done = bars + 12;           // 1
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = p.cluster;
    const uint32_t rank = c > 1 ? cluster_ctarank() : 0u;
    const uint16_t all = (uint16_t)((1u << c) - 1u);
    const int b = blockIdx.y;
    const int q0 = blockIdx.x * TQ;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(q_full), 1);
        for (int s = 0; s < KV_STAGES; ++s) {
            mbar_init(smem_u32(&k_full[s]), (uint32_t)c);    // one arm per issuer of a slice
            mbar_init(smem_u32(&v_full[s]), (uint32_t)c);
            mbar_init(smem_u32(&kv_empty[s]), (uint32_t)c);  // one release per consumer CTA
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_empty[i]), 4);
        }
        mbar_init(smem_u32(p_full), 4);
        mbar_init(smem_u32(pv_done), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), 512);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    if (c > 1) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;        // columns: S0 [0,128), S1 [128,256), O [256,384)

    if ((warp == 0 || warp == 6) && lane == 0) {
        // ---------------------------------------------------------------- producers
        const bool is_k = warp == 0;
        const CUtensorMap* tm = is_k ? &tmK : &tmV;
        prefetch_tmap(tm);
        if (is_k) {
            prefetch_tmap(&tmQ);
            mbar_arrive_expect_tx_local(smem_u32(q_full), TILE_BYTES);
            tma_load_4d(smem_u32(sQ), &tmQ, smem_u32(q_full), 0, q0, 0, b);
        }
        // This CTA's slice of each shared tile. K (K-major, 2 atoms): whole atoms
        // first, then rows within an atom. V (MN-major, 2 boxes of 64 d columns x 128
        // keys): a band of key rows of both boxes.
        int atom0 = 0, r0 = 0, rows = TK;
        if (is_k) {
            if (c <= 2) { atom0 = (int)rank; }
            else { atom0 = (int)rank / (c / 2); r0 = ((int)rank % (c / 2)) * (TK / (c / 2)); }
        } else {
            rows = TK / c;
            r0 = (int)rank * rows;
        }
        const uint32_t slice_bytes = TILE_BYTES / (uint32_t)c;
        uint64_t* full = is_k ? k_full : v_full;
        uint8_t* base = is_k ? sK : sV;
        for (int j = 0; j < p.n_kv; ++j) {
            const int s = j % KV_STAGES;
            const uint32_t ph = (uint32_t)(j / KV_STAGES) & 1u;
            if (!attn_wait(smem_u32(&kv_empty[s]), ph ^ 1u, p, 1)) break;
            const uint32_t fb = smem_u32(&full[s]);
            for (int r = 0; r < c; ++r) {
                if (r == (int)rank) mbar_arrive_expect_tx_local(fb, slice_bytes);
                else mbar_arrive_expect_tx_cluster(mapa(fb, (uint32_t)r), slice_bytes);
            }
            const uint32_t tile = smem_u32(base + s * TILE_BYTES);
            const int key0 = j * TK;
            if (is_k) {
                const uint32_t dst = tile + (uint32_t)(atom0 * ATOM_BYTES + r0 * 128);
                if (c > 1) tma_load_4d_mcast(dst, tm, fb, 0, key0 + r0, atom0, b, all);
                else       tma_load_4d(dst, tm, fb, 0, key0 + r0, 0, b);
            } else {
                for (int box = 0; box < HD / 64; ++box) {
                    const uint32_t dst = tile + (uint32_t)(box * TK * 128 + r0 * 128);
                    if (c > 1) tma_load_3d_mcast(dst, tm, fb, box * 64, key0 + r0, b, all);
                    else       tma_load_3d(dst, tm, fb, box * 64, key0 + r0, b);
                }
            }
        }
        // Every stage this thread filled is released by all receivers before exit.
        for (int j = p.n_kv; j < p.n_kv + KV_STAGES; ++j) {
            const int s = j % KV_STAGES;
            if (!attn_wait(smem_u32(&kv_empty[s]), ((uint32_t)(j / KV_STAGES) & 1u) ^ 1u, p, 1)) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t idesc_s = instr_desc_bf16(TQ, TK, false, false);    // Q (K-major) x K^T (K-major)
        const uint32_t idesc_o = instr_desc_bf16(TQ, HD, false, true);     // P (K-major) x V (MN-major)
        const uint64_t dq = smem_desc_sw128(smem_u32(sQ), false, 0);
        const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), false, 0);
        const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), true, TK * 128);
        const uint64_t dp = smem_desc_sw128(smem_u32(sP), false, 0);
        const uint16_t release_mask = all;
        bool ok = attn_wait(smem_u32(q_full), 0, p, 2);
        auto issue_s = [&](int j) -> bool {
            const int s = j % KV_STAGES;
            if (!attn_wait(smem_u32(&k_full[s]), (uint32_t)(j / KV_STAGES) & 1u, p, 3)) return false;
            const int sb = j & 1;
            if (!attn_wait(smem_u32(&s_empty[sb]), ((uint32_t)(j >> 1) & 1u) ^ 1u, p, 4)) return false;
            tc_fence_after();
            const uint64_t dk = dk0 + ((s * TILE_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < HD / 16; ++k)
                mma_bf16<1>(tmem + sb * TK, dq + kmajor_koff(k), dk + kmajor_koff(k), idesc_s, k > 0 ? 1u : 0u);
            mma_commit<1>(smem_u32(&s_full[sb]));
            return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 0; ok && j < p.n_kv; ++j) {
            if (j + 1 < p.n_kv && !issue_s(j + 1)) { ok = false; break; }
            const int s = j % KV_STAGES;
            if (!attn_wait(smem_u32(p_full), (uint32_t)j & 1u, p, 5)) { ok = false; break; }
            if (!attn_wait(smem_u32(&v_full[s]), (uint32_t)(j / KV_STAGES) & 1u, p, 6)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dv = dv0 + ((s * TILE_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < TK / 16; ++k)
                mma_bf16<1>(tmem + 2 * TK, dp + kmajor_koff(k), dv + mnmajor_koff(k), idesc_o,
                            (j > 0 || k > 0) ? 1u : 0u);
            mma_commit<1>(smem_u32(pv_done));
            // K_j and V_j are consumed: release the stage to every CTA that fills it.
            if (c > 1) mma_commit_mcast<1>(smem_u32(&kv_empty[s]), release_mask);
            else       mma_commit<1>(smem_u32(&kv_empty[s]));
        }
        (void)ok;
    } else if (warp >= 2 && warp <= 5) {
        // ---------------------------------------------------------------- softmax
        const int qd = warp & 3;                     // TMEM lane quadrant
        const int row = qd * 32 + lane;              // query row within the tile
        const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
        float m_ref = -INFINITY;                     // reference max, base-2 units
        float l = 0.0f;                              // running sum of exp2(x - m_ref)
        bool ok = true;
        for (int j = 0; j < p.n_kv; ++j) {
            const int sb = j & 1;
            if (!attn_wait(smem_u32(&s_full[sb]), (uint32_t)(j >> 1) & 1u, p, 7)) { ok = false; break; }
            tc_fence_after();
            float x[TK];
#pragma unroll
            for (int cchunk = 0; cchunk < TK / 32; ++cchunk) {
                uint32_t r[32];
                tmem_ld_32cols(lane_base + sb * TK + cchunk * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) x[cchunk * 32 + i] = __uint_as_float(r[i]) * p.scale_log2;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(smem_u32(&s_empty[sb]));
            const int valid = p.sk - j * TK;         // keys of this tile inside the sequence
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < TK; ++i) {
                if (i >= valid) x[i] = -INFINITY;
                mx = fmaxf(mx, x[i]);
            }
            float alpha = 1.0f;                      // factor for O and l when the reference moves
            if (j == 0) {
                m_ref = mx;
            } else if (mx > m_ref + RESCALE_THRESHOLD) {
                alpha = exp2f(m_ref - mx);
                m_ref = mx;
            }
            l *= alpha;
            uint32_t pk[TK / 2];
#pragma unroll
            for (int i = 0; i < TK / 2; ++i) {
                const float p0 = exp2f(x[2 * i] - m_ref);
                const float p1 = exp2f(x[2 * i + 1] - m_ref);
                l += p0 + p1;
                pk[i] = pack_bf16x2(p0, p1);
            }
            if (j > 0) {
                // P_{j-1} V_{j-1} has completed: O is stable and the P buffer is free.
                if (!attn_wait(smem_u32(pv_done), (uint32_t)(j - 1) & 1u, p, 8)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                    for (int cchunk = 0; cchunk < HD / 32; ++cchunk) {
                        uint32_t r[32];
                        const uint32_t ta = lane_base + 2 * TK + cchunk * 32;
                        tmem_ld_32cols(ta, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st_32cols(ta, r);
                    }
                    tmem_st_wait();
                }
            }
            // P row into the K-major swizzled A-operand tile: keys 0-63 in atom 0, 64-127 in atom 1;
            // 16-byte chunk g of row r sits at chunk g ^ (r % 8).
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                uint8_t* rowp = sP + a * ATOM_BYTES + row * 128;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int w = a * 32 + g * 4;
                    *reinterpret_cast<uint4*>(rowp + ((g ^ (row & 7)) << 4)) =
                        make_uint4(pk[w], pk[w + 1], pk[w + 2], pk[w + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_local(smem_u32(p_full));
        }
        // Final normalisation: O / l, and lse = (m_ref + log2 l) * ln 2.
        if (ok && attn_wait(smem_u32(pv_done), (uint32_t)(p.n_kv - 1) & 1u, p, 9)) {
            tc_fence_after();
            const int q = q0 + row;
            const float inv = 1.0f / l;
            for (int cchunk = 0; cchunk < HD / 32; ++cchunk) {
                uint32_t r[32];
                tmem_ld_32cols(lane_base + 2 * TK + cchunk * 32, r);
                tmem_ld_wait();
                if (q < p.sq) {
                    const long long off = ((long long)b * p.sq + q) * HD + cchunk * 32;
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
        tmem_dealloc<1>(tmem, 512);
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
                                               int out_f32, int cluster, void* stream) {
    if (batch < 0 || sq < 0 || sk < 0) return afail(GEMM_ERR_INVALID_ARG, "negative size");
    if (batch == 0 || sq == 0) return GEMM_OK;
    if (sk == 0) return afail(GEMM_ERR_INVALID_ARG, "sk must be at least 1");
    if (d != HD) return afail(GEMM_ERR_UNSUPPORTED, "head dimension must be 128");
    if (cluster != 1 && cluster != 2 && cluster != 4) return afail(GEMM_ERR_UNSUPPORTED, "cluster must be 1, 2 or 4");
    if (!Q || !K || !V || !O) return afail(GEMM_ERR_INVALID_ARG, "null pointer");
    if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) |
         reinterpret_cast<uintptr_t>(O) | reinterpret_cast<uintptr_t>(lse)) & 15u)
        return afail(GEMM_ERR_ALIGNMENT, "Q, K, V, O and lse must be 16-byte aligned");
    if (batch >= 65536 || sq >= (1ll << 31) || sk >= (1ll << 31)) return afail(GEMM_ERR_INVALID_ARG, "too large");
    auto enc = attn_encoder();
    if (!enc) return afail(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    CUtensorMap tq, tk, tv;
    // Q and K: the k-split view {64, rows, 2 atoms, batch} (atoms 128 bytes apart).
    const cuuint64_t qd[4] = {64, (cuuint64_t)sq, 2, (cuuint64_t)batch};
    const cuuint64_t qs[3] = {HD * 2, 128, (cuuint64_t)(sq * HD * 2)};
    const cuuint32_t qb[4] = {64, TQ, 2, 1};
    const cuuint64_t kd[4] = {64, (cuuint64_t)sk, 2, (cuuint64_t)batch};
    const cuuint64_t ks[3] = {HD * 2, 128, (cuuint64_t)(sk * HD * 2)};
    // A K slice: whole atoms first (cluster <= 2), then half the rows of one atom (cluster 4).
    const cuuint32_t kb[4] = {64, (cuuint32_t)(cluster <= 2 ? TK : TK / 2), (cuuint32_t)(cluster == 1 ? 2 : 1), 1};
    // V: MN-major boxes of 64 d columns x (128 / cluster) keys.
    const cuuint64_t vd[3] = {HD, (cuuint64_t)sk, (cuuint64_t)batch};
    const cuuint64_t vs[2] = {HD * 2, (cuuint64_t)(sk * HD * 2)};
    const cuuint32_t vb[3] = {64, (cuuint32_t)(TK / cluster), 1};
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
    const size_t smem = 1024 + 6 * TILE_BYTES + 14 * 8 + 16;
    void* fn = reinterpret_cast<void*>(&attention_fwd_kernel);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return afail(GEMM_ERR_CUDA, cudaGetErrorString(e));
    long long qtiles = (sq + TQ - 1) / TQ;
    qtiles = (qtiles + cluster - 1) / cluster * cluster;    // whole clusters; extra tiles store nothing
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)qtiles, (unsigned)batch, 1);
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
    snprintf(g_attn_err, sizeof g_attn_err, "attention: bounded wait %u expired (q tile %u, batch %u)", w[0], w[1], w[2]);
    return GEMM_ERR_DEVICE_TIMEOUT;
}
