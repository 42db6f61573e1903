// attn_tc.cuh -- sparse absorbed-MLA attention on the sm_103a tensor cores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the main MLA
// attention is computed only over the index_topk selected tokens (the
// additive-mask formulation, exact because exp(-inf) = 0).  Absorbed form at
// the DeepseekV32Config sizes: 128 heads, query/key width 576 = latent 512
// (kv_lora_rank) + rope 64 (qk_rope_head_dim), value = the 512-d latent.
//
// One query per CLUSTER OF TWO CTAs.  The fp32 output O[128 x 512] alone
// fills a CTA's whole tensor memory (512 columns x 128 lanes x 4 B), so the
// pair splits the latent between them:
//   rank 0 owns key columns 0..255 and the rope columns 512..575,
//   rank 1 owns key columns 256..511;
// each rank gathers only its columns of the selected rows (no byte of a row
// is fetched twice), computes a PARTIAL score tile S_r = Q_r . K_r^T over
// its columns, and the two partials are exchanged through distributed
// shared memory so both hold S = S_0 + S_1 (fp32 addition commutes, so both
// hold identical S and take identical softmax decisions).  Each rank then
// accumulates O[:, its 256 latent columns] += P . V_r, where V_r is exactly
// the latent part of the columns it gathered.  No flop is duplicated.
//
// Per CTA (288 threads):
//   warps 0..3  softmax: one head (TMEM lane) per thread; exchange, online
//               softmax with a lazily updated running max (O is rescaled
//               only when the max grows by more than 2^8), P (bf16) to
//               shared memory, final 1/l scaling and the output store;
//   warp 4      TMEM allocation and tcgen05.mma issue (one thread);
//   warps 5..8  gather: cp.async of the selected rows (16 B per copy) into
//               128B-swizzled tiles, 32 keys per block, 4-stage ring.
// TMEM: two S buffers (32 columns each) and O (256 columns).
#pragma once

#include <cuda.h>

#include "rows.cuh"

namespace dsa {

constexpr int kAttnHeads = 128;
constexpr int kAttnDqk = 576;
constexpr int kAttnDv = 512;
constexpr int kAttnBK = 32;              // selected keys per block
constexpr int kAttnStages = 4;           // gather ring depth
constexpr int kAttnThreads = 288;
constexpr int kAttnMaxSlots = 5;         // 64-column slots per rank (rank 0: 5, rank 1: 4)

struct AttnTc {
    static constexpr int Q_SLOT = kAttnHeads * 128;                 // 128 heads x 64 cols bf16 = 16 KB
    static constexpr int KV_SLOT = kAttnBK * 128;                   // 32 keys x 64 cols = 4 KB
    static constexpr int KV_STAGE = kAttnMaxSlots * KV_SLOT;        // 20 KB
    static constexpr int P_BUF = kAttnHeads * 128;                  // 128 rows x 128 B (first 64 B used)
    static constexpr int X_BUF = kAttnHeads * kAttnBK * 4;          // peer's partial scores, 16 KB
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_KV = OFF_Q + kAttnMaxSlots * Q_SLOT;
    static constexpr int OFF_P = OFF_KV + kAttnStages * KV_STAGE;
    static constexpr int OFF_X = OFF_P + 2 * P_BUF;
    static constexpr int OFF_BAR = OFF_X + X_BUF;
    // barriers: q_full, kv_full[4], kv_empty[4], s_full[2], p_full[2], pv_done[2], x_full, x_free, done
    static constexpr int NBAR = 1 + 2 * kAttnStages + 2 + 2 + 2 + 3;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;
    static constexpr int TMEM_COLS = 512;
    static constexpr int TM_S = 0;        // S buffers at columns 0 and 32
    static constexpr int TM_O = 256;      // O at columns 256..511
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, kAttnBK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);
};

__device__ __forceinline__ int attn_slot_kblock(int rank, int j) {
    // rank 0: latent blocks 0..3 then the rope block 8; rank 1: latent blocks 4..7
    return rank == 0 ? (j < 4 ? j : 8) : 4 + j;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __nv_bfloat16* __restrict__ kv,
               const int* __restrict__ idx, RowSpec rs, int k, float scale_log2, __nv_bfloat16* __restrict__ out,
               float* __restrict__ lse, unsigned long long timeout_ns) {
    using C = AttnTc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sKV = sbase + C::OFF_KV, sP = sbase + C::OFF_P, sX = sbase + C::OFF_X;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    const uint32_t q_full = bar0;
    auto kv_full = [&](int i) { return bar0 + 8u * (1 + i); };
    auto kv_empty = [&](int i) { return bar0 + 8u * (1 + kAttnStages + i); };
    auto s_full = [&](int i) { return bar0 + 8u * (1 + 2 * kAttnStages + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (3 + 2 * kAttnStages + i); };
    auto pv_done = [&](int i) { return bar0 + 8u * (5 + 2 * kAttnStages + i); };
    const uint32_t x_full = bar0 + 8u * (7 + 2 * kAttnStages);
    const uint32_t x_free = bar0 + 8u * (8 + 2 * kAttnStages);
    const uint32_t done_bar = bar0 + 8u * (9 + 2 * kAttnStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int peer = rank ^ 1;
    const int r = blockIdx.x >> 1;                 // query row of this cluster
    const int nslot = (rank == 0) ? 5 : 4;

    const RowInfo ri = row_info(rs, r);
    const int nsel = ri.ok ? min(k, ri.n) : 0;     // valid entries of the index row
    const int nb = (nsel + kAttnBK - 1) / kAttnBK;
    const int* irow = idx + static_cast<long long>(r) * k;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kAttnStages; ++i) { mbar_init(kv_full(i), 128); mbar_init(kv_empty(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(p_full(i), 128); mbar_init(pv_done(i), 1); }
        mbar_init(x_full, 128);
        mbar_init(x_free, 128);
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();             // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 4) {
        if (lane == 0 && nb > 0) {
            // ---------------- Q load + MMA issue ----------------
            mbar_expect_tx(q_full, nslot * C::Q_SLOT);
            for (int j = 0; j < nslot; ++j)
                tma_load_2d(sQ + j * C::Q_SLOT, &tm_q, attn_slot_kblock(rank, j) * 64, r * kAttnHeads, q_full);
            bool ok = wait_bar(q_full, 0, timeout_ns, s_abort);
            auto issue_qk = [&](int i) -> bool {
                const int st = i % kAttnStages;
                if (!wait_bar(kv_full(st), (i / kAttnStages) & 1, timeout_ns, s_abort)) return false;
                tc_fence_after();
                const uint32_t d = tmem_base + C::TM_S + (i & 1) * kAttnBK;
                for (int j = 0; j < nslot; ++j) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t a = sdesc_sw128(sQ + j * C::Q_SLOT + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(sKV + st * C::KV_STAGE + j * C::KV_SLOT + kk * 32, 16, 1024);
                        tc_mma_bf16(d, a, b, C::IDESC_QK, (j | kk) ? 1u : 0u);
                    }
                }
                tc_commit(s_full(i & 1));
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int i = 0; i < nb && ok; ++i) {
                if (i + 1 < nb) ok = issue_qk(i + 1);
                if (!ok) break;
                ok = wait_bar(p_full(i & 1), (i >> 1) & 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const int st = i % kAttnStages;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {   // K = 32 keys = 2 x 16
                    const uint64_t a = sdesc_sw128(sP + (i & 1) * C::P_BUF + kk * 32, 16, 1024);
                    // V (MN-major): 64-column chunks are the 4 latent slots (LBO), 8-key groups 1 KB apart (SBO)
                    const uint64_t b = sdesc_sw128(sKV + st * C::KV_STAGE + kk * 16 * 128, C::KV_SLOT, 1024);
                    tc_mma_bf16(tmem_base + C::TM_O, a, b, C::IDESC_PV, (i | kk) ? 1u : 0u);
                }
                tc_commit(pv_done(i & 1));
                tc_commit(kv_empty(st));
            }
            tc_commit(done_bar);
            wait_bar(done_bar, 0, timeout_ns, nullptr);
        }
    } else if (warp >= 5) {
        // ---------------- gather producers ----------------
        const int p = tid - 5 * 32;                  // 0..127
        const int chunks_per_key = nslot * 8;
        const int nchunks = kAttnBK * chunks_per_key;
        bool ok = true;
        for (int i = 0; i < nb && ok; ++i) {
            const int st = i % kAttnStages;
            ok = wait_bar(kv_empty(st), ((i / kAttnStages) & 1) ^ 1, timeout_ns, s_abort);
            if (!ok) break;
            const uint32_t stage = sKV + st * C::KV_STAGE;
            for (int id = p; id < nchunks; id += 128) {
                const int kk = id / chunks_per_key;
                const int rem = id - kk * chunks_per_key;
                const int j = rem >> 3, c = rem & 7;
                const int e = i * kAttnBK + kk;
                int s = (e < nsel) ? __ldg(irow + e) : 0;
                if (s < 0 || s >= ri.n) {
                    if (e < nsel) raise_error(DSA_ERR_DEVICE_DATA);
                    s = 0;   // any in-range row; columns past nsel are masked by the softmax
                }
                const __nv_bfloat16* src = kv + (ri.key_base + s) * kAttnDqk + attn_slot_kblock(rank, j) * 64 + c * 8;
                cp_async_16(stage + j * C::KV_SLOT + sw128_off(kk, c), src);
            }
            cp_async_commit();
            if (i > 0) {   // block i-1 has landed: publish it (one block stays in flight)
                cp_async_wait<1>();
                fence_proxy_async_smem();
                mbar_arrive(kv_full((i - 1) % kAttnStages));
            }
        }
        if (ok && nb > 0) {
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(kv_full((nb - 1) % kAttnStages));
        } else {
            cp_async_wait<0>();
        }
    } else {
        // ---------------- softmax / output (warps 0..3) ----------------
        const int h = warp * 32 + lane;              // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t x_full_peer = mapa(x_full, peer), x_free_peer = mapa(x_free, peer);
        const uint32_t sX_peer = mapa(sX, peer);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nb && ok; ++i) {
            const int b = i & 1;
            ok = __all_sync(0xffffffffu, wait_bar(s_full(b), (i >> 1) & 1, timeout_ns, s_abort));
            if (!ok) break;
            tc_fence_after();
            uint32_t sraw[32];
            tmem_ld32(tmem_base + lane_off + C::TM_S + b * kAttnBK, sraw);
            tmem_ld_wait();
            // exchange the partial scores with the peer CTA
            ok = __all_sync(0xffffffffu, wait_bar<true>(x_free, (i & 1) ^ 1, timeout_ns, s_abort));
            if (!ok) break;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_cluster_v4(sX_peer + h * 128 + (((c ^ h) & 7) << 4), __uint_as_float(sraw[4 * c]),
                              __uint_as_float(sraw[4 * c + 1]), __uint_as_float(sraw[4 * c + 2]),
                              __uint_as_float(sraw[4 * c + 3]));
            mbar_arrive_cluster(x_full_peer);
            ok = __all_sync(0xffffffffu, wait_bar<true>(x_full, i & 1, timeout_ns, s_abort));
            if (!ok) break;
            float sv[32];
            const float4* xr = reinterpret_cast<const float4*>(smem + C::OFF_X + h * 128);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = xr[(c ^ h) & 7];
                sv[4 * c + 0] = __uint_as_float(sraw[4 * c + 0]) + v.x;
                sv[4 * c + 1] = __uint_as_float(sraw[4 * c + 1]) + v.y;
                sv[4 * c + 2] = __uint_as_float(sraw[4 * c + 2]) + v.z;
                sv[4 * c + 3] = __uint_as_float(sraw[4 * c + 3]) + v.w;
            }
            mbar_arrive_cluster(x_free_peer);
            // columns past the last valid entry are masked (identical for every head)
            const int nvalid = nsel - i * kAttnBK;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                sv[j] = (j < nvalid) ? sv[j] * scale_log2 : -INFINITY;
                mx = fmaxf(mx, sv[j]);
            }
            const float m_new = fmaxf(m, mx);
            const bool resc = m_new > m + 8.f;           // lazy rescale (always true on the first block)
            const float factor = resc ? fast_exp2(m - m_new) : 1.f;
            if (i > 0 && __any_sync(0xffffffffu, resc)) {
                // O must hold every earlier P.V before it is rescaled
                ok = __all_sync(0xffffffffu,
                                wait_bar(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1, timeout_ns, s_abort));
                if (!ok) break;
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tmem_base + lane_off + C::TM_O + c0, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * factor);
                    tmem_st32(tmem_base + lane_off + C::TM_O + c0, o);
                }
                tmem_st_wait();
            }
            if (resc) {
                l *= factor;
                m = m_new;
            }
            // P = 2^(z - m) in bf16; l sums the rounded values that the MMA uses
            uint32_t pk[16];
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(fast_exp2(sv[2 * j] - m), fast_exp2(sv[2 * j + 1] - m));
                const float2 back = __bfloat1622float2(pr);
                lsum += back.x + back.y;
                pk[j] = *reinterpret_cast<const uint32_t*>(&pr);
            }
            l += lsum;
            if (i >= 2) {   // P buffer b was read by P.V of block i-2
                ok = __all_sync(0xffffffffu, wait_bar(pv_done(b), ((i - 2) >> 1) & 1, timeout_ns, s_abort));
                if (!ok) break;
            }
            uint8_t* prow = smem + C::OFF_P + b * C::P_BUF;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(prow + sw128_off(h, c)) =
                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full(b));
        }
        // ---------------- epilogue ----------------
        const long long orow = (static_cast<long long>(r) * kAttnHeads + h) * kAttnDv + rank * 256;
        if (ok && nb > 0) {
            ok = __all_sync(0xffffffffu,
                            wait_bar(pv_done((nb - 1) & 1), ((nb - 1) >> 1) & 1, timeout_ns, s_abort));
            if (ok) {
                tc_fence_after();
                const float inv = 1.f / l;
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(tmem_base + lane_off + C::TM_O + c0, o);
                    tmem_ld_wait();
                    uint4* dst = reinterpret_cast<uint4*>(out + orow + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                                                           __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
                            pk[e] = *reinterpret_cast<const uint32_t*>(&v);
                        }
                        dst[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                if (lse != nullptr && rank == 0)
                    lse[static_cast<long long>(r) * kAttnHeads + h] = (m + log2f(l)) * 0.69314718055994530942f;
            }
        } else if (nb == 0) {   // no valid selection (invalid row): zeros, lse = -inf
            uint4* dst = reinterpret_cast<uint4*>(out + orow);
            for (int q = 0; q < 32; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr && rank == 0) lse[static_cast<long long>(r) * kAttnHeads + h] = -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();             // the peer no longer writes into this CTA's shared memory
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace dsa
