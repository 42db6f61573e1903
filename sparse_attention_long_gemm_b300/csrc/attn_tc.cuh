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
//
// Shared memory is mostly a 4-slot ring.  Its items, in the order every role
// walks them: per query, one Q item (two slots: the latent part of Q_r in
// four 128B-swizzled 16 KB tiles and the rope part in two 64B-swizzled 4 KB
// halves, loaded by TMA), then one KV item per 64-key block (one slot: the
// rank's 288 columns of the 64 selected rows, latent 128B-swizzled, rope
// 64B-swizzled).  The softmax warps move a Q item into tensor memory (latent)
// and a small rope buffer, freeing its slots at once, so nearly the whole ring
// holds gathers in flight: random rows reach about 9 TB/s from L2 only with
// ~100 KB per SM in flight and with requests of 512 contiguous bytes.
//
// Per CTA (224 threads):
//   warps 0..3  softmax: one head (TMEM lane) per thread; Q items into
//               tensor memory, the score exchange (each thread stores its
//               row of partial scores locally, then one bulk copy moves the
//               32 KB tile into the peer CTA and completes the peer's
//               mbarrier: single 16-byte remote stores reach only ~7 B/clk),
//               the online softmax
//               with a lazily updated running max (O is rescaled only when the
//               max grows by more than 2^8), P into tensor memory, and the
//               output epilogue;
//   warp 4      TMEM allocation and tcgen05.mma issue (one thread);
//   warps 5..6  producers: the rows of a KV item by cp.async, each warp
//               instruction one key's 512 latent bytes (the rope parts of 8
//               keys per instruction), completion signalled with
//               cp.async.mbarrier.arrive.noinc so the producers never wait for
//               data; index loads run four blocks ahead; one thread issues the
//               TMA loads of Q items.
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
constexpr int kAttnSlots = 4;            // ring slots
constexpr int kAttnThreads = 224;
constexpr int kAttnProducers = 64;       // threads of warps 5..6

struct AttnTc {
    static constexpr int KV_SLOT = kAttnBK * 128;                   // 64 keys x 64 latent cols = 8 KB
    static constexpr int KV_ROPE = kAttnBK * 64;                    // 64 keys x 32 rope cols = 4 KB
    static constexpr int SLOT = 4 * KV_SLOT + KV_ROPE;              // 36 KB
    static constexpr int QL_TILE = kAttnHeads * 128;                // 128 heads x 64 latent cols = 16 KB
    static constexpr int QR_HALF = 64 * 64;                         // 64 heads x 32 rope cols = 4 KB
    static constexpr int QR_BYTES = 2 * QR_HALF;
    static constexpr int X_BYTES = kAttnHeads * kAttnBK * 4;        // peer's partial scores, 32 KB
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_QR = OFF_RING + kAttnSlots * SLOT;
    static constexpr int OFF_X = OFF_QR + QR_BYTES;                 // the peer's partial scores land here
    static constexpr int OFF_XS = OFF_X + X_BYTES;                  // this CTA's partial scores, sent in bulk
    static constexpr int OFF_BAR = OFF_XS + X_BYTES;
    // full[S], empty[S], q_tm_full, s_full[2], p_full[2], pv_done[2], x_full, x_free, done
    static constexpr int NBAR = 2 * kAttnSlots + 1 + 2 + 2 + 2 + 3;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;               // + alignment slack
    static constexpr int TMEM_COLS = 512;
    static constexpr int TM_O = 0;
    static constexpr int TM_Q = 256;
    static constexpr int TM_SP = 384;     // + 64 * buffer
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, kAttnBK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);
    static constexpr uint32_t Q_TX = 4 * QL_TILE + QR_BYTES;
};
static_assert(AttnTc::SMEM <= 232448, "attention shared memory exceeds the per-CTA limit");
static_assert(2 * AttnTc::QL_TILE + AttnTc::QR_HALF <= AttnTc::SLOT, "a Q item must fit in two slots");

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

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory into
// another CTA's (address from mapa); completes `bytes` on that CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t rdst, uint32_t src, uint32_t bytes, uint32_t rbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(rdst), "r"(src), "r"(bytes), "r"(rbar) : "memory");
}

// Arrive on `bar` once every cp.async issued so far by this thread has landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
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
               const __nv_bfloat16* __restrict__ kv, const int* __restrict__ idx, RowSpec rs, int rows, int k,
               float scale_log2, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
               unsigned long long timeout_ns) {
    using C = AttnTc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sRing = sbase + C::OFF_RING, sQR = sbase + C::OFF_QR, sX = sbase + C::OFF_X;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kAttnSlots + i); };
    const uint32_t q_tm_full = bar0 + 8u * (2 * kAttnSlots);
    auto s_full = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 1 + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 3 + i); };
    auto pv_done = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 5 + i); };
    const uint32_t x_full = bar0 + 8u * (2 * kAttnSlots + 7);
    const uint32_t x_free = bar0 + 8u * (2 * kAttnSlots + 8);
    const uint32_t done_bar = bar0 + 8u * (2 * kAttnSlots + 9);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    auto slot_addr = [&](int rp) { return sRing + static_cast<uint32_t>(rp % kAttnSlots) * C::SLOT; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int peer = rank ^ 1;
    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;

    if (tid == 0) {
        for (int i = 0; i < kAttnSlots; ++i) { mbar_init(full(i), kAttnProducers); mbar_init(empty(i), 1); }
        mbar_init(q_tm_full, 128);
        for (int i = 0; i < 2; ++i) { mbar_init(s_full(i), 1); mbar_init(p_full(i), 128); mbar_init(pv_done(i), 1); }
        mbar_init(x_full, 1);       // the local expect_tx; the peer's bytes complete it
        mbar_init(x_free, 4);       // one arrive per softmax warp of the peer
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_q_rope);
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

    if (warp >= 5) {
        // ---------------- producers: Q items (TMA) and KV items (cp.async) ----------------
        const int pt = tid - 5 * 32;                 // 0..63
        const int pw = pt >> 5;                      // which half of the block's keys
        int rp = 0;
        bool ok = true;
        for (int r = cl; r < rows && ok; r += ncl) {
            const AttnRow A = attn_row(rs, r, k);
            if (A.nb == 0) continue;
            // Q item: two slots
            ok = wait_bar(empty(rp % kAttnSlots), ((rp / kAttnSlots) & 1) ^ 1, timeout_ns, s_abort) &&
                 wait_bar(empty((rp + 1) % kAttnSlots), (((rp + 1) / kAttnSlots) & 1) ^ 1, timeout_ns, s_abort);
            if (!ok) break;
            if (pt == 0) {
                const uint32_t fb = full(rp % kAttnSlots);
                mbar_expect_tx(fb, C::Q_TX);
                for (int j = 0; j < 4; ++j)
                    tma_load_2d(slot_addr(rp + (j >> 1)) + (j & 1) * C::QL_TILE, &tm_q, rank * 256 + j * 64,
                                r * kAttnHeads, fb);
                for (int hh = 0; hh < 2; ++hh)
                    tma_load_2d(slot_addr(rp + hh) + 2 * C::QL_TILE, &tm_q_rope, 512 + rank * 32,
                                r * kAttnHeads + hh * 64, fb);
            } else {
                mbar_arrive(full(rp % kAttnSlots));
            }
            mbar_arrive(full((rp + 1) % kAttnSlots));
            rp += 2;
            // KV items
            const int* irow = idx + static_cast<long long>(r) * k;
            const long long kb = A.ri.key_base;
            const int kown = pw * 32 + lane;         // key of the block whose index this thread loads
            int e0, e1, e2, e3;
            auto ld_ent = [&](int i) {
                const int ent = i * kAttnBK + kown;
                return (ent < A.nsel) ? __ldg(irow + ent) : 0;
            };
            e0 = ld_ent(0); e1 = ld_ent(1); e2 = ld_ent(2); e3 = ld_ent(3);
            for (int i = 0; i < A.nb && ok; ++i, ++rp) {
                int s = e0;
                if (s < 0 || s >= A.ri.n) {
                    if (i * kAttnBK + kown < A.nsel) raise_error(DSA_ERR_DEVICE_DATA);
                    s = 0;   // any in-range row; entries past nsel are masked by the softmax
                }
                const long long myrow = kb + s;
                e0 = e1; e1 = e2; e2 = e3; e3 = ld_ent(i + 4);
                ok = wait_bar(empty(rp % kAttnSlots), ((rp / kAttnSlots) & 1) ^ 1, timeout_ns, s_abort);
                if (!ok) break;
                const uint32_t st = slot_addr(rp);
                // latent: one key (512 contiguous bytes) per warp instruction
                const int j = lane >> 3, c = lane & 7;
#pragma unroll 8
                for (int kk = 0; kk < 32; ++kk) {
                    const long long row = __shfl_sync(0xffffffffu, myrow, kk);
                    const int key = pw * 32 + kk;
                    cp_async_16(st + j * C::KV_SLOT + key * 128 + (((c ^ key) & 7) << 4),
                                kv + row * kAttnDqk + rank * 256 + lane * 8);
                }
                // rope: 8 keys (64 bytes each) per warp instruction
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int kl = t * 8 + (lane >> 2), cc = lane & 3;
                    const long long row = __shfl_sync(0xffffffffu, myrow, kl);
                    const int key = pw * 32 + kl;
                    cp_async_16(st + 4 * C::KV_SLOT + key * 64 + (((cc ^ (key >> 1)) & 3) << 4),
                                kv + row * kAttnDqk + 512 + rank * 32 + cc * 8);
                }
                cp_async_arrive_noinc(full(rp % kAttnSlots));
            }
        }
        cp_async_wait<0>();
        if (!ok) sleep_ns(2000000ull);  // let copies already issued land before the CTA exits
    } else if (warp == 4) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int qi = 0, gi = 0, rp = 0;
            bool ok = true;
            const uint64_t dQR = sdesc_sw64(sQR);                          // Q rope part
            // ring slot rp: keys (latent, K-major), keys (rope), values (MN-major)
            auto dK = [&](int rp_) { return sdesc_sw128(slot_addr(rp_), 16, 1024); };
            auto dR = [&](int rp_) { return sdesc_sw64(slot_addr(rp_) + 4 * C::KV_SLOT); };
            auto dV = [&](int rp_) { return sdesc_sw128(slot_addr(rp_), C::KV_SLOT, 1024); };
            auto issue_qk = [&](int g, int rp_) -> bool {
                if (!wait_bar(full(rp_ % kAttnSlots), (rp_ / kAttnSlots) & 1, timeout_ns, s_abort)) return false;
                fence_proxy_async_smem();   // rows written by cp.async, read by the tensor cores
                tc_fence_after();
                const uint32_t d = tmem_base + C::TM_SP + (g & 1) * kAttnBK;
                const uint64_t bk = dK(rp_), br = dR(rp_);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_ts(d, tmem_base + C::TM_Q + j * 32 + kk * 8,
                                       bk + static_cast<uint64_t>((j * C::KV_SLOT + kk * 32) >> 4), C::IDESC_QK,
                                       (j | kk) ? 1u : 0u);
                }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    tc_mma_bf16(d, dQR + static_cast<uint64_t>(kk * 2), br + static_cast<uint64_t>(kk * 2),
                                C::IDESC_QK, 1u);
                tc_commit(s_full(g & 1));
                return true;
            };
            for (int r = cl; r < rows && ok; r += ncl) {
                const AttnRow A = attn_row(rs, r, k);
                if (A.nb == 0) continue;
                rp += 2;                                   // the Q item (consumed by the softmax warps)
                ok = wait_bar(q_tm_full, qi & 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const int g0 = gi, rp0 = rp;
                ok = issue_qk(g0, rp0);
                if (ok && A.nb > 1) ok = issue_qk(g0 + 1, rp0 + 1);
                for (int i = 0; i < A.nb && ok; ++i) {
                    const int g = g0 + i;
                    ok = wait_bar(p_full(g & 1), (g >> 1) & 1, timeout_ns, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t bv = dV(rp0 + i);
#pragma unroll
                    for (int kk = 0; kk < kAttnBK / 16; ++kk)
                        // V (MN-major): the 4 latent slots are the 64-column chunks (LBO), 8-key groups 1 KB apart
                        tc_mma_bf16_ts(tmem_base + C::TM_O, tmem_base + C::TM_SP + (g & 1) * kAttnBK + kk * 8,
                                       bv + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::IDESC_PV,
                                       (i | kk) ? 1u : 0u);
                    tc_commit(pv_done(g & 1));
                    tc_commit(empty((rp0 + i) % kAttnSlots));
                    if (i + 2 < A.nb) ok = issue_qk(g + 2, rp0 + i + 2);
                }
                gi = g0 + A.nb;
                rp = rp0 + A.nb;
                ++qi;
            }
            tc_commit(done_bar);                          // every MMA issued has completed
            wait_bar(done_bar, 0, timeout_ns, nullptr);   // before TMEM is released
        }
    } else {
        // ---------------- softmax / Q items / epilogue (warps 0..3) ----------------
        const int h = warp * 32 + lane;              // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t x_full_peer = mapa(x_full, peer), x_free_peer = mapa(x_free, peer);
        const uint32_t sX_peer = mapa(sX, peer);
        const uint8_t* xrow = smem + C::OFF_X + h * 256;
        uint8_t* xsrow = smem + C::OFF_XS + h * 256;
        int qi = 0, gi = 0, rp = 0;
        bool ok = true;

        // Moves the Q item at ring position rp_ into tensor memory (latent) and the rope buffer.
        auto take_q = [&](int rp_) -> bool {
            const int sa = rp_ % kAttnSlots, sb = (rp_ + 1) % kAttnSlots;
            if (!__all_sync(0xffffffffu, wait_bar(full(sa), (rp_ / kAttnSlots) & 1, timeout_ns, s_abort) &&
                                             wait_bar(full(sb), ((rp_ + 1) / kAttnSlots) & 1, timeout_ns, s_abort)))
                return false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t v[32];
                const uint8_t* src = smem + C::OFF_RING + ((rp_ + (j >> 1)) % kAttnSlots) * C::SLOT +
                                     (j & 1) * C::QL_TILE + h * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4*>(src + (((c ^ h) & 7) << 4));
                    v[4 * c + 0] = u.x; v[4 * c + 1] = u.y; v[4 * c + 2] = u.z; v[4 * c + 3] = u.w;
                }
                tmem_st32(tmem_base + lane_off + C::TM_Q + j * 32, v);
            }
            {   // rope rows keep their byte offsets, so the 64-byte swizzle is preserved
                const uint8_t* src = smem + C::OFF_RING + ((rp_ + (h >> 6)) % kAttnSlots) * C::SLOT + 2 * C::QL_TILE +
                                     (h & 63) * 64;
                uint4* dst = reinterpret_cast<uint4*>(smem + C::OFF_QR + h * 64);
#pragma unroll
                for (int c = 0; c < 4; ++c) dst[c] = reinterpret_cast<const uint4*>(src)[c];
            }
            fence_proxy_async_smem();
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(q_tm_full);
            named_sync(1, 128);                       // every thread has read the item
            if (h == 0) {
                mbar_arrive(empty(sa));
                mbar_arrive(empty(sb));
            }
            return true;
        };
        auto zero_row = [&](int rr) {   // no valid selection (invalid row): zeros, lse = -inf
            uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<long long>(rr) * kAttnHeads + h) * kAttnDv + rank * 256);
            for (int q = 0; q < 32; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
            if (lse != nullptr && rank == 0) lse[static_cast<long long>(rr) * kAttnHeads + h] = -INFINITY;
        };

        // the first query with work
        int r = cl;
        AttnRow A;
        while (r < rows) {
            A = attn_row(rs, r, k);
            if (A.nb > 0) break;
            zero_row(r);
            r += ncl;
        }
        if (r < rows) {
            ok = take_q(rp);
            rp += 2;
        }
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
                // exchange the partial scores with the peer CTA.  x_free: the peer has read
                // the previous tile, so the previous bulk copy out of XS has completed too.
                ok = __all_sync(0xffffffffu, wait_bar<true>(x_free, (g & 1) ^ 1, timeout_ns, s_abort));
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4*>(xsrow + (((c ^ h) & 15) << 4)) =
                        make_uint4(sraw[4 * c], sraw[4 * c + 1], sraw[4 * c + 2], sraw[4 * c + 3]);
                fence_proxy_async_smem();
                named_sync(1, 128);
                if (h == 0) {
                    mbar_expect_tx(x_full, C::X_BYTES);
                    bulk_copy_to_peer(sX_peer, sbase + C::OFF_XS, C::X_BYTES, x_full_peer);
                }
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
            rp += A.nb;
            const int r_cur = r;
            // next query with work; its Q goes into tensor memory now (every Q.K^T of this
            // query has completed: the last s_full was observed above)
            r += ncl;
            while (r < rows) {
                A = attn_row(rs, r, k);
                if (A.nb > 0) break;
                zero_row(r);
                r += ncl;
            }
            ++qi;
            if (r < rows) {
                ok = take_q(rp);
                rp += 2;
            }
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
            if (lse != nullptr && rank == 0)
                lse[static_cast<long long>(r_cur) * kAttnHeads + h] = (m + log2f(l)) * 0.69314718055994530942f;
            tc_fence_before();   // O has been read before the next query's first P.V overwrites it
        }
        (void)qi;
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
