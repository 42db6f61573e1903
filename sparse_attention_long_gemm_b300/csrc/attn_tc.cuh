// attn_tc.cuh -- sparse absorbed-MLA attention on the sm_103a tensor cores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the main MLA
// attention is computed only over the index_topk selected tokens (the
// additive-mask formulation, exact because exp(-inf) = 0).  Absorbed form at
// the DeepseekV32Config sizes: 128 heads, query/key width 576 = latent 512
// (kv_lora_rank) + rope 64 (qk_rope_head_dim), value = the 512-d latent.
//
// One query at a time per CLUSTER OF TWO CTAs; the kernel is persistent
// (cluster c takes rows c, c + #clusters, ...).  The fp32 output
// O[128 x 512] alone would fill a CTA's whole tensor memory, so the pair
// splits the key/value columns:
//   rank r owns latent columns 256r .. 256r+255 and rope columns
//   512+32r .. 512+32r+31 (288 of the 576 contraction columns each).
// Each rank gathers only its columns of the selected rows (no byte of a row
// is fetched twice), computes a PARTIAL score tile S_r = Q_r . K_r^T over its
// columns, and the two partials are exchanged through distributed shared
// memory so both hold S = S_0 + S_1 (fp32 addition commutes, so both hold
// bit-identical S and take identical softmax decisions).  Each rank then
// accumulates O[:, its 256 latent columns] += P . V_r, where V_r is the
// latent part of the columns it gathered.  No flop is duplicated.
//
// Tensor memory of a CTA (512 columns x 128 lanes, lane = head):
//   [0, 256)    O_r, fp32 accumulator
//   [256, 384)  Q_r latent part, bf16 pairs: the A operand of Q.K^T
//   [384, 448)  S/P buffer 0: fp32 partial scores of a 64-key block, then
//               (after the exchange) the bf16 probabilities P over its first
//               32 columns, which are the A operand of P.V
//   [448, 512)  S/P buffer 1
// Keeping Q and P in tensor memory leaves shared-memory bandwidth to the
// gathered keys and the score exchange.
//
// Per CTA (192 threads):
//   warp 0      producer: TMA loads of Q (latent part to a staging buffer,
//               rope part in place) and TMA gather4 of the selected rows
//               (4 rows per instruction) into a 3-stage ring of 64-key
//               blocks, latent columns 128B-swizzled, rope 64B-swizzled;
//   warp 1      TMEM allocation and tcgen05.mma issue (one thread);
//   warps 2..5  softmax: one head (TMEM lane) per thread; the exchange, the
//               online softmax with a lazily updated running max (O is
//               rescaled only when the max grows by more than 2^8), P into
//               tensor memory, copying the next query's Q into tensor
//               memory, and the output epilogue.
// MMA order per query: QK(0), QK(1), PV(0), QK(2), PV(1), QK(3), ...; a
// QK(i+2) reuses the S/P buffer of PV(i), which is safe because tcgen05
// operations issued by one thread execute in order.
#pragma once

#include <cuda.h>

#include "rows.cuh"

namespace dsa {

constexpr int kAttnHeads = 128;
constexpr int kAttnDqk = 576;
constexpr int kAttnDv = 512;
constexpr int kAttnBK = 64;              // selected keys per block
constexpr int kAttnStages = 3;           // gather ring depth
constexpr int kAttnThreads = 192;

struct AttnTc {
    static constexpr int QL_SLOT = kAttnHeads * 128;                // 128 heads x 64 latent cols bf16 = 16 KB
    static constexpr int QL_BYTES = 4 * QL_SLOT;                    // 64 KB staging
    static constexpr int QR_BYTES = kAttnHeads * 64;                // 128 heads x 32 rope cols = 8 KB
    static constexpr int KV_SLOT = kAttnBK * 128;                   // 64 keys x 64 latent cols = 8 KB
    static constexpr int KV_ROPE = kAttnBK * 64;                    // 64 keys x 32 rope cols = 4 KB
    static constexpr int KV_STAGE = 4 * KV_SLOT + KV_ROPE;          // 36 KB
    static constexpr int X_BYTES = kAttnHeads * kAttnBK * 4;        // peer's partial scores, 32 KB
    static constexpr int OFF_QL = 0;
    static constexpr int OFF_QR = OFF_QL + QL_BYTES;
    static constexpr int OFF_KV = OFF_QR + 2 * QR_BYTES;
    static constexpr int OFF_X = OFF_KV + kAttnStages * KV_STAGE;
    static constexpr int OFF_BAR = OFF_X + X_BYTES;
    // q_full[2], q_tm_full, q_stage_free, rope_free[2], kv_full[S], kv_empty[S],
    // s_full[2], p_full[2], pv_done[2], x_full, x_free, done
    static constexpr int NBAR = 2 + 1 + 1 + 2 + 2 * kAttnStages + 2 + 2 + 2 + 3;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;               // + alignment slack
    static constexpr int TMEM_COLS = 512;
    static constexpr int TM_O = 0;
    static constexpr int TM_Q = 256;
    static constexpr int TM_SP = 384;     // + 64 * buffer
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, kAttnBK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);
    static constexpr uint32_t Q_TX = QL_BYTES + QR_BYTES;
    static constexpr uint32_t KV_TX = KV_STAGE;
};
static_assert(AttnTc::SMEM <= 232448, "attention shared memory exceeds the per-CTA limit");

// Shared-memory matrix descriptor, 64-byte-swizzled K-major operand
// (rows of 64 B, 8-row atoms of 512 B).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (unused when swizzled)
    d |= static_cast<uint64_t>(512 >> 4) << 32;                // next 8-row group
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(4) << 61;                       // 64-byte swizzle
    return d;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 with A read from tensor memory
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// TMA gather of 4 whole rows (row coordinates r0..r3) of a 2-D tensor, box
// columns starting at column x, into consecutive box rows at dst.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap, int x, int r0, int r1, int r2, int r3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

// Asynchronous store of 16 bytes into another CTA's shared memory (address
// from mapa); completes `bytes` on that CTA's mbarrier (also from mapa).
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(raddr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(rbar) : "memory");
}

// Rows of one query: number of valid selected entries and of 64-key blocks.
struct AttnRow {
    RowInfo ri;
    int nsel;
    int nb;
};
__device__ __forceinline__ AttnRow attn_row(const RowSpec& rs, int r, int k) {
    AttnRow a;
    a.ri = row_info(rs, r);
    a.nsel = a.ri.ok ? min(k, a.ri.n) : 0;
    a.nb = (a.nsel + kAttnBK - 1) / kAttnBK;
    return a;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q_rope,
               const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kv_rope,
               const int* __restrict__ idx, RowSpec rs, int rows, int k, float scale_log2,
               __nv_bfloat16* __restrict__ out, float* __restrict__ lse, unsigned long long timeout_ns) {
    using C = AttnTc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQL = sbase + C::OFF_QL, sQR = sbase + C::OFF_QR, sKV = sbase + C::OFF_KV;
    const uint32_t sX = sbase + C::OFF_X;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto q_full = [&](int i) { return bar0 + 8u * i; };
    const uint32_t q_tm_full = bar0 + 8u * 2;
    const uint32_t q_stage_free = bar0 + 8u * 3;
    auto rope_free = [&](int i) { return bar0 + 8u * (4 + i); };
    auto kv_full = [&](int i) { return bar0 + 8u * (6 + i); };
    auto kv_empty = [&](int i) { return bar0 + 8u * (6 + kAttnStages + i); };
    auto s_full = [&](int i) { return bar0 + 8u * (6 + 2 * kAttnStages + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (8 + 2 * kAttnStages + i); };
    auto pv_done = [&](int i) { return bar0 + 8u * (10 + 2 * kAttnStages + i); };
    const uint32_t x_full = bar0 + 8u * (12 + 2 * kAttnStages);
    const uint32_t x_free = bar0 + 8u * (13 + 2 * kAttnStages);
    const uint32_t done_bar = bar0 + 8u * (14 + 2 * kAttnStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int peer = rank ^ 1;
    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) { mbar_init(q_full(i), 1); mbar_init(rope_free(i), 1); }
        mbar_init(q_tm_full, 128);
        mbar_init(q_stage_free, 128);
        for (int i = 0; i < kAttnStages; ++i) { mbar_init(kv_full(i), 1); mbar_init(kv_empty(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(p_full(i), 128); mbar_init(pv_done(i), 1); }
        mbar_init(x_full, 1);       // the local expect_tx; the peer's bytes complete it
        mbar_init(x_free, 4);       // one arrive per softmax warp of the peer
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_q_rope);
        tma_prefetch_desc(&tm_kv);
        tma_prefetch_desc(&tm_kv_rope);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();             // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: Q loads and row gathers ----------------
        int qi = 0, gi = 0;
        bool ok = true;
        for (int r = cl; r < rows && ok; r += ncl) {
            const AttnRow A = attn_row(rs, r, k);
            if (A.nb == 0) continue;
            if (lane == 0) {
                ok = wait_bar(q_stage_free, (qi & 1) ^ 1, timeout_ns, s_abort) &&
                     wait_bar(rope_free(qi & 1), ((qi >> 1) & 1) ^ 1, timeout_ns, s_abort);
                if (ok) {
                    const uint32_t qb = q_full(qi & 1);
                    mbar_expect_tx(qb, C::Q_TX);
                    for (int j = 0; j < 4; ++j)
                        tma_load_2d(sQL + j * C::QL_SLOT, &tm_q, rank * 256 + j * 64, r * kAttnHeads, qb);
                    tma_load_2d(sQR + (qi & 1) * C::QR_BYTES, &tm_q_rope, 512 + rank * 32, r * kAttnHeads, qb);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            const int* irow = idx + static_cast<long long>(r) * k;
            const int kb = static_cast<int>(A.ri.key_base);
            // this lane's 4 entries of block i (lanes 0..15 cover the 64 keys); loads run
            // three blocks ahead of their use so their latency hides behind the ring
            auto load_ent = [&](int i, int (&v)[4]) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int ent = i * kAttnBK + 4 * (lane & 15) + e;
                    v[e] = (ent < A.nsel) ? __ldg(irow + ent) : 0;
                }
            };
            int e0[4], e1[4], e2[4];
            load_ent(0, e0);
            load_ent(1, e1);
            load_ent(2, e2);
            for (int i = 0; i < A.nb && ok; ++i, ++gi) {
                const int st = gi % kAttnStages;
                int rw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int ent = i * kAttnBK + 4 * (lane & 15) + e;
                    int s = e0[e];
                    if (s < 0 || s >= A.ri.n) {
                        if (ent < A.nsel) raise_error(DSA_ERR_DEVICE_DATA);
                        s = 0;   // any in-range row; entries past nsel are masked by the softmax
                    }
                    rw[e] = kb + s;
                    e0[e] = e1[e];
                    e1[e] = e2[e];
                }
                load_ent(i + 3, e2);
                if (lane == 0) {
                    ok = wait_bar(kv_empty(st), ((gi / kAttnStages) & 1) ^ 1, timeout_ns, s_abort);
                    if (ok) mbar_expect_tx(kv_full(st), C::KV_TX);
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (lane < 16) {
                    const uint32_t stage = sKV + st * C::KV_STAGE;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_gather4(stage + j * C::KV_SLOT + lane * 512, &tm_kv, rank * 256 + j * 64, rw[0], rw[1],
                                    rw[2], rw[3], kv_full(st));
                    tma_gather4(stage + 4 * C::KV_SLOT + lane * 256, &tm_kv_rope, 512 + rank * 32, rw[0], rw[1],
                                rw[2], rw[3], kv_full(st));
                }
                __syncwarp();
            }
            ++qi;
        }
        if (!ok) sleep_ns(2000000ull);  // let copies already issued land before the CTA exits
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int qi = 0, gi = 0;
            bool ok = true;
            // descriptors of stage 0 / rope buffer 0; other stages and K-steps are offsets
            // of the start-address field (16-byte units)
            const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);              // keys, latent slots (K-major)
            const uint64_t dR0 = sdesc_sw64(sKV + 4 * C::KV_SLOT);        // keys, rope part
            const uint64_t dV0 = sdesc_sw128(sKV, C::KV_SLOT, 1024);      // values (MN-major)
            const uint64_t dQR0 = sdesc_sw64(sQR);                        // Q rope part
            auto issue_qk = [&](int g, int qb) -> bool {
                const int st = g % kAttnStages;
                if (!wait_bar(kv_full(st), (g / kAttnStages) & 1, timeout_ns, s_abort)) return false;
                tc_fence_after();
                const uint32_t d = tmem_base + C::TM_SP + (g & 1) * kAttnBK;
                const uint64_t so = static_cast<uint64_t>((st * C::KV_STAGE) >> 4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_ts(d, tmem_base + C::TM_Q + j * 32 + kk * 8,
                                       dK0 + so + static_cast<uint64_t>((j * C::KV_SLOT + kk * 32) >> 4), C::IDESC_QK,
                                       (j | kk) ? 1u : 0u);
                }
                const uint64_t qo = static_cast<uint64_t>((qb * C::QR_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    tc_mma_bf16(d, dQR0 + qo + static_cast<uint64_t>(kk * 2), dR0 + so + static_cast<uint64_t>(kk * 2),
                                C::IDESC_QK, 1u);
                tc_commit(s_full(g & 1));
                return true;
            };
            for (int r = cl; r < rows && ok; r += ncl) {
                const AttnRow A = attn_row(rs, r, k);
                if (A.nb == 0) continue;
                const int qb = qi & 1;
                ok = wait_bar(q_full(qb), (qi >> 1) & 1, timeout_ns, s_abort) &&
                     wait_bar(q_tm_full, qi & 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const int g0 = gi;
                ok = issue_qk(g0, qb);
                if (ok && A.nb > 1) ok = issue_qk(g0 + 1, qb);
                for (int i = 0; i < A.nb && ok; ++i) {
                    const int g = g0 + i;
                    ok = wait_bar(p_full(g & 1), (g >> 1) & 1, timeout_ns, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    const int st = g % kAttnStages;
                    const uint64_t so = static_cast<uint64_t>((st * C::KV_STAGE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kAttnBK / 16; ++kk)
                        // V (MN-major): the 4 latent slots are the 64-column chunks (LBO), 8-key groups 1 KB apart
                        tc_mma_bf16_ts(tmem_base + C::TM_O, tmem_base + C::TM_SP + (g & 1) * kAttnBK + kk * 8,
                                       dV0 + so + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::IDESC_PV,
                                       (i | kk) ? 1u : 0u);
                    tc_commit(pv_done(g & 1));
                    tc_commit(kv_empty(st));
                    if (i + 2 < A.nb) ok = issue_qk(g + 2, qb);
                }
                tc_commit(rope_free(qb));
                gi = g0 + A.nb;
                ++qi;
            }
            tc_commit(done_bar);                          // every MMA issued has completed
            wait_bar(done_bar, 0, timeout_ns, nullptr);   // before TMEM is released
        }
    } else {
        // ---------------- softmax / Q copy / epilogue (warps 2..5) ----------------
        const int quad = warp & 3;
        const int h = quad * 32 + lane;              // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t x_full_peer = mapa(x_full, peer), x_free_peer = mapa(x_free, peer);
        const uint32_t sX_peer = mapa(sX, peer);
        const uint8_t* xrow = smem + C::OFF_X + h * 256;
        int qi = 0, gi = 0;
        bool ok = true;

        // Copies Q (latent part, staged by TMA) of the qi-th processed query into tensor memory.
        auto copy_q = [&](int qj) -> bool {
            if (!__all_sync(0xffffffffu, wait_bar(q_full(qj & 1), (qj >> 1) & 1, timeout_ns, s_abort))) return false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t v[32];
                const uint8_t* src = smem + C::OFF_QL + j * C::QL_SLOT + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src + (((c ^ h) & 7) << 4));
                    v[4 * c + 0] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
                }
                tmem_st32(tmem_base + lane_off + C::TM_Q + j * 32, v);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(q_tm_full);
            mbar_arrive(q_stage_free);
            return true;
        };

        // the first query with work
        int r = cl;
        AttnRow A;
        while (r < rows) {
            A = attn_row(rs, r, k);
            if (A.nb > 0) break;
            // no valid selection (invalid row): zeros, lse = -inf
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<long long>(r) * kAttnHeads + h) * kAttnDv + rank * 256);
            for (int q = 0; q < 32; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr && rank == 0) lse[static_cast<long long>(r) * kAttnHeads + h] = -INFINITY;
            r += ncl;
        }
        if (r < rows) ok = copy_q(0);
        while (r < rows && ok) {
            float m = -INFINITY, l = 0.f;
            const int g0 = gi;
            for (int i = 0; i < A.nb && ok; ++i) {
                const int g = g0 + i, b = g & 1;
                ok = __all_sync(0xffffffffu, wait_bar(s_full(b), (g >> 1) & 1, timeout_ns, s_abort));
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[64];
                tmem_ld32(tmem_base + lane_off + C::TM_SP + b * kAttnBK, *reinterpret_cast<uint32_t(*)[32]>(sraw));
                tmem_ld32(tmem_base + lane_off + C::TM_SP + b * kAttnBK + 32,
                          *reinterpret_cast<uint32_t(*)[32]>(sraw + 32));
                tmem_ld_wait();
                // exchange the partial scores with the peer CTA: asynchronous remote stores
                // that complete the peer's x_full transaction count
                ok = __all_sync(0xffffffffu, wait_bar<true>(x_free, (g & 1) ^ 1, timeout_ns, s_abort));
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    st_async_v4(sX_peer + h * 256 + (((c ^ h) & 15) << 4), sraw[4 * c], sraw[4 * c + 1], sraw[4 * c + 2],
                                sraw[4 * c + 3], x_full_peer);
                if (h == 0) mbar_expect_tx(x_full, C::X_BYTES);
                ok = __all_sync(0xffffffffu, wait_bar<true>(x_full, g & 1, timeout_ns, s_abort));
                if (!ok) break;
                float sv[64];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 v = *reinterpret_cast<const float4*>(xrow + (((c ^ h) & 15) << 4));
                    sv[4 * c + 0] = __uint_as_float(sraw[4 * c + 0]) + v.x;
                    sv[4 * c + 1] = __uint_as_float(sraw[4 * c + 1]) + v.y;
                    sv[4 * c + 2] = __uint_as_float(sraw[4 * c + 2]) + v.z;
                    sv[4 * c + 3] = __uint_as_float(sraw[4 * c + 3]) + v.w;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(x_free_peer);   // this warp's rows of X may be overwritten
                // columns past the last valid entry are masked (identical for every head)
                const int nvalid = A.nsel - i * kAttnBK;
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    sv[j] = (j < nvalid) ? sv[j] * scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sv[j]);
                }
                const float m_new = fmaxf(m, mx);
                const bool resc = m_new > m + 8.f;           // lazy rescale (always true on the first block)
                const float factor = resc ? fast_exp2(m - m_new) : 1.f;
                if (i > 0 && __any_sync(0xffffffffu, resc)) {
                    // O must hold every earlier P.V before it is rescaled
                    ok = __all_sync(0xffffffffu,
                                    wait_bar(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1, timeout_ns, s_abort));
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
                }
                if (resc) {
                    l *= factor;
                    m = m_new;
                }
                // P = 2^(z - m) in bf16 (pairs of keys per 32-bit column); l sums the rounded values
                uint32_t pk[32];
                float lsum = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const __nv_bfloat162 pr = __floats2bfloat162_rn(fast_exp2(sv[2 * j] - m), fast_exp2(sv[2 * j + 1] - m));
                    const float2 back = __bfloat1622float2(pr);
                    lsum += back.x + back.y;
                    pk[j] = *reinterpret_cast<const uint32_t*>(&pr);
                }
                l += lsum;
                tmem_st32(tmem_base + lane_off + C::TM_SP + b * kAttnBK, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_full(b));
            }
            if (!ok) break;
            gi = g0 + A.nb;
            const int r_cur = r;
            const int nb_cur = A.nb;
            // next query with work; its Q goes into tensor memory now (every Q.K^T of this
            // query has completed: the last s_full was observed above)
            r += ncl;
            while (r < rows) {
                A = attn_row(rs, r, k);
                if (A.nb > 0) break;
                uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<long long>(r) * kAttnHeads + h) * kAttnDv + rank * 256);
                for (int q = 0; q < 32; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
                if (lse != nullptr && rank == 0) lse[static_cast<long long>(r) * kAttnHeads + h] = -INFINITY;
                r += ncl;
            }
            ++qi;
            if (r < rows) ok = copy_q(qi);
            // ---------------- epilogue of the finished query ----------------
            const int gl = gi - 1;
            ok = ok && __all_sync(0xffffffffu, wait_bar(pv_done(gl & 1), (gl >> 1) & 1, timeout_ns, s_abort));
            if (!ok) break;
            tc_fence_after();
            const float inv = 1.f / l;
            const long long orow = (static_cast<long long>(r_cur) * kAttnHeads + h) * kAttnDv + rank * 256;
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
            (void)nb_cur;
            if (lse != nullptr && rank == 0)
                lse[static_cast<long long>(r_cur) * kAttnHeads + h] = (m + log2f(l)) * 0.69314718055994530942f;
            tc_fence_before();   // O has been read before the next query's first P.V overwrites it
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();             // the peer no longer writes into this CTA's shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace dsa
