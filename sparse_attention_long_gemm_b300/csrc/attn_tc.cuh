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
// is fetched twice) and computes PARTIAL scores S_r = Q_r . K_r^T for all 128
// heads over its columns.  The softmax of a head is owned by one rank: rank r
// owns heads 64r .. 64r+63.  Per 64-key block each rank sends the peer its
// partial scores of the peer's heads (16 KB, fp32) and receives the peer's
// partial scores of its own heads; it completes S = S_0 + S_1 for its heads,
// runs their online softmax, and writes their probabilities P (bf16) straight
// into its half of a 128-head P tile in shared memory, the A operand of P.V.
// The same 8 KB half is bulk-copied into the peer's P tile, together with each
// head's O rescale factor and softmax denominator (512 B).  Both ranks then
// hold P for all 128 heads and accumulate O[:, their 256 latent columns] +=
// P . V_r.  No flop is duplicated, and 24.5 KB per block cross between the
// CTAs in each direction (distributed shared memory moves ~14.5 B/clk per SM).
//
// Tensor memory of a CTA (512 columns x 128 lanes, lane = head):
//   [0, 256)    O_r, fp32 accumulator
//   [256, 384)  Q_r latent part, bf16 pairs: the A operand of Q.K^T
//   [384, 512)  S buffers 0 and 1: fp32 partial scores of a 64-key block.
//               Two buffers let the tensor cores run the Q.K^T of later
//               blocks while the softmax of the current one waits for the
//               exchange, so the exchange of a block overlaps the softmax of
//               the block before it.
//
// Shared memory is mostly a 4-slot ring.  Its items, in the order every role
// walks them: per query, one Q item (two slots: the latent part of Q_r in
// four 128B-swizzled 16 KB tiles and the rope part in two 64B-swizzled 4 KB
// halves, loaded by TMA), then one KV item per 64-key block (one slot: the
// rank's 288 columns of the 64 selected rows, latent 128B-swizzled, rope
// 64B-swizzled).  The softmax warps move a Q item into tensor memory (latent)
// and a small rope buffer, freeing its slots at once, so nearly the whole ring
// holds gathers in flight: random rows reach about 9 TB/s from L2 only with
// ~100 KB per SM in flight and with requests of 512 contiguous bytes.  The
// rest holds the two P tiles (128B-swizzled, K-major), the received partial
// scores (one 16 KB buffer, returned to the sender as soon as the owning warps
// have loaded it), an 8 KB staging buffer per sending warp (its 32 heads, one
// bulk copy per block) and the rescale factors / denominators (two buffers
// each way).
//
// Per CTA (256 threads; the warp of a role depends on the rank so that the two
// warps running the softmax have their SM sub-partitions to themselves):
//   warps 0..3  softmax group, one head (TMEM lane) per thread.  The two
//               warps whose lanes are this rank's heads ("own" warps)
//               complete their scores, run the online softmax (running max
//               updated lazily: O is rescaled only when it grows by more than
//               2^8) and write their half of the P tile; the two others
//               ("peer" warps) send their lanes' partial scores and take the
//               rescale factors that come with the peer's half of P
//               (rescaling those O rows first when told to).  Each peer warp
//               polls both jobs with non-blocking barrier tests, sending as
//               soon as a block's S is in and the peer's buffer is free and
//               taking whenever the peer's P has arrived (staging the next
//               block's scores when neither is ready), so neither stream
//               waits behind the other.  All four move Q items into tensor
//               memory and run the output epilogue;
//   one warp    copy warp (warp 4 on rank 0, warp 6 on rank 1): one thread
//               sends this rank's half of each P tile, with its factors, to
//               the peer by bulk copy as soon as the own warps have written
//               it and the peer has freed its copy, so the own warps never
//               wait for the peer;
//   one warp    TMEM allocation and tcgen05.mma issue (one thread, polling
//               both the next Q.K^T and the next P.V so neither waits on the
//               other; after each P.V it also returns the peer's P receive
//               buffer with a multicast tcgen05.commit): warp 6 on rank 0,
//               warp 4 on rank 1;
//   two warps   producers (warps 5 and 7), each gathering half of the keys of
//               every KV item by cp.async: each warp instruction one key's 512
//               latent bytes (the rope parts of 8 keys per instruction),
//               completion signalled with cp.async.mbarrier.arrive.noinc so the
//               producers never wait for data; index loads run four blocks
//               ahead; one thread issues the TMA loads of Q items.
#pragma once

#include <cuda.h>

#include "rows.cuh"

namespace dsa {

constexpr int kAttnHeads = 128;
constexpr int kAttnDqk = 576;
constexpr int kAttnDv = 512;
constexpr int kAttnBK = 64;              // selected keys per block
constexpr int kAttnSlots = 4;            // ring slots
constexpr int kAttnThreads = 256;
constexpr int kAttnProducers = 64;       // threads of the two producer warps

struct AttnTc {
    static constexpr int KV_SLOT = kAttnBK * 128;                   // 64 keys x 64 latent cols = 8 KB
    static constexpr int KV_ROPE = kAttnBK * 64;                    // 64 keys x 32 rope cols = 4 KB
    static constexpr int SLOT = 4 * KV_SLOT + KV_ROPE;              // 36 KB
    static constexpr int QL_TILE = kAttnHeads * 128;                // 128 heads x 64 latent cols = 16 KB
    static constexpr int QR_HALF = 64 * 64;                         // 64 heads x 32 rope cols = 4 KB
    static constexpr int QR_BYTES = 2 * QR_HALF;
    static constexpr int XB = 64 * kAttnBK * 4;                     // partial scores of 64 heads: 16 KB
    static constexpr int XSW = 32 * kAttnBK * 4;                    // one peer warp's staging: 32 heads, 8 KB
    static constexpr int PT = kAttnHeads * kAttnBK * 2;             // P tile of 128 heads: 16 KB
    static constexpr int PH = PT / 2;                               // one rank's 64 heads of it
    static constexpr int MB = 64 * 4 * 2;                           // rescale factors + denominators
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_QR = OFF_RING + kAttnSlots * SLOT;
    static constexpr int OFF_P = OFF_QR + QR_BYTES;                 // [2] P tiles
    static constexpr int OFF_XR = OFF_P + 2 * PT;                   // received partial scores
    static constexpr int OFF_XS = OFF_XR + XB;                      // [2 peer warps] outgoing partial scores
    static constexpr int OFF_MR = OFF_XS + 2 * XSW;                 // [2] received factors / denominators
    static constexpr int OFF_MS = OFF_MR + 2 * MB;                  // [2] outgoing factors / denominators
    static constexpr int OFF_BAR = OFF_MS + 2 * MB;
    // full[S], empty[S], q_tm_full, s_full[2], s_free[2], p_full[2], pv_done[2],
    // xr_full, xr_free, pr_full[2], pr_free[2], done, p_ready[2], pcopy_done[2]
    static constexpr int NBAR = 2 * kAttnSlots + 1 + 2 + 2 + 2 + 2 + 1 + 1 + 2 + 2 + 1 + 2 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int USED = OFF_MISC + 16;
    // Slack for aligning the dynamic shared memory base to 1024 bytes (the 128B-swizzled
    // operands need it): whatever the per-CTA limit leaves.  The base is 1024-aligned in
    // practice; a launch whose base needs more padding reports an error and computes nothing.
    static constexpr int SLACK = (232448 - USED) < 1024 ? (232448 - USED) : 1024;
    static constexpr int SMEM = USED + SLACK;
    static constexpr int TMEM_COLS = 512;
    static constexpr int TM_O = 0;
    static constexpr int TM_Q = 256;
    static constexpr int TM_S = 384;      // + 64 * buffer
    static constexpr uint32_t IDESC_QK = idesc_bf16(128, kAttnBK, false, false);
    static constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);
    static constexpr uint32_t Q_TX = 4 * QL_TILE + QR_BYTES;
    static constexpr uint32_t P_TX = PH + MB;                       // bytes of one P message
};
static_assert(AttnTc::SMEM <= 232448, "attention shared memory exceeds the per-CTA limit");
static_assert(AttnTc::OFF_P % 1024 == 0, "the P tiles are 128B-swizzled operands (1024-byte atoms)");
static_assert(2 * AttnTc::QL_TILE + AttnTc::QR_HALF <= AttnTc::SLOT, "a Q item must fit in two slots");
static_assert(AttnTc::SLACK >= 0, "attention shared memory exceeds the per-CTA limit");
static_assert(AttnTc::PH % 16 == 0 && AttnTc::MB % 16 == 0 && AttnTc::XB % 16 == 0 && AttnTc::XSW % 16 == 0,
              "bulk copies move multiples of 16 bytes");

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
// bulk_commit() closes this thread's current bulk async-group.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t rdst, uint32_t src, uint32_t bytes, uint32_t rbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(rdst), "r"(src), "r"(bytes), "r"(rbar) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's most recent bulk async-groups still read their sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Arrive on `bar` once every cp.async issued so far by this thread has landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Relaxed arrive on an mbarrier of the peer CTA that cannot be performed
// before the shared-memory loads behind `dep` have returned their data.  The
// caller ORs bits of every loaded value into `dep`; `zero` is 0 at run time
// but opaque to the compiler (derived from a kernel argument), so the address
// remote_bar + (dep & zero) truly depends on the loaded registers and the
// arrive waits for them.  A warp-wide load completes for all of its lanes at
// once, so one lane's dependency covers the warp's loads of the same
// instructions.  This hands a receive buffer back to the peer without the
// cost of a cluster-scope release.
__device__ __forceinline__ void mbar_arrive_cluster_after(uint32_t remote_bar, uint32_t dep, uint32_t zero) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar + (dep & zero))
                 : "memory");
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

// PAGED: the selected rows come from paged pools through the block table of `rs`.
template <bool PAGED = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q_rope,
               const __nv_bfloat16* __restrict__ kv, const int* __restrict__ idx, RowSpec rs, int rows, int k,
               float scale_log2, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
               unsigned long long timeout_ns) {
    using C = AttnTc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (smem - smem_raw > C::SLACK) {   // uniform over the grid: every CTA has the same base
        if (threadIdx.x == 0) raise_error(DSA_ERR_UNSUPPORTED);
        return;
    }
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sRing = sbase + C::OFF_RING, sQR = sbase + C::OFF_QR;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto full = [&](int i) { return bar0 + 8u * i; };
    auto empty = [&](int i) { return bar0 + 8u * (kAttnSlots + i); };
    const uint32_t q_tm_full = bar0 + 8u * (2 * kAttnSlots);
    auto s_full = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 1 + i); };
    auto s_free = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 3 + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 5 + i); };
    auto pv_done = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 7 + i); };
    const uint32_t xr_full = bar0 + 8u * (2 * kAttnSlots + 9);
    const uint32_t xr_free = bar0 + 8u * (2 * kAttnSlots + 10);
    auto pr_full = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 11 + i); };
    auto pr_free = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 13 + i); };
    const uint32_t done_bar = bar0 + 8u * (2 * kAttnSlots + 15);
    auto p_ready = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 16 + i); };
    auto pcopy_done = [&](int i) { return bar0 + 8u * (2 * kAttnSlots + 18 + i); };
    const uint32_t sP = sbase + C::OFF_P;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    auto slot_addr = [&](int rp) { return sRing + static_cast<uint32_t>(rp % kAttnSlots) * C::SLOT; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const uint32_t opaque_zero = static_cast<uint32_t>(rows) >> 31;   // rows >= 0: always 0
    const int peer = rank ^ 1;
    const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    // Warps w and w+4 share an SM sub-partition; the softmax ("own") warps are 0,1 on rank 0
    // and 2,3 on rank 1, so the MMA and producer warps go to the other two sub-partitions.
    const int mma_warp = (rank == 0) ? 6 : 4;
    const int prod_warp = (rank == 0) ? 7 : 5;
    const int copy_warp = (rank == 0) ? 4 : 6;
    const int prod_warp2 = (rank == 0) ? 5 : 7;

    if (tid == 0) {
        for (int i = 0; i < kAttnSlots; ++i) { mbar_init(full(i), kAttnProducers); mbar_init(empty(i), 1); }
        mbar_init(q_tm_full, 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(s_free(i), 128);
            mbar_init(p_full(i), 128);
            mbar_init(pv_done(i), 1);
            mbar_init(pr_full(i), 1);     // a local expect_tx; the peer's bulk copies complete it
            mbar_init(pr_free(i), 1);     // the peer's MMA thread: its P.V of the buffer has completed
            mbar_init(p_ready(i), 2);     // one arrive per own warp: its rows of P and factors are written
            mbar_init(pcopy_done(i), 1);  // the copy warp: this rank's half has been read by its copy
        }
        mbar_init(xr_full, 1);            // a local expect_tx; the peer's two bulk copies complete it
        mbar_init(xr_free, 2);            // one arrive per own warp of the peer
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_q_rope);
    }
    if (warp == mma_warp) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();             // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == prod_warp || warp == prod_warp2) {
        // ---------------- producers: Q items (TMA) and KV items (cp.async) ----------------
        // Each warp gathers half of every block's keys (keys 32 pw .. 32 pw + 31).
        const int pw = (warp == prod_warp) ? 0 : 1;
        int rp = 0;
        bool ok = true;
        for (int r = cl; r < rows && ok; r += ncl) {
            const AttnRow A = attn_row(rs, r, k);
            if (A.nb == 0) continue;
            // Q item: two slots
            ok = wait_bar(empty(rp % kAttnSlots), ((rp / kAttnSlots) & 1) ^ 1, timeout_ns, s_abort) &&
                 wait_bar(empty((rp + 1) % kAttnSlots), (((rp + 1) / kAttnSlots) & 1) ^ 1, timeout_ns, s_abort);
            if (!ok) break;
            if (pw == 0 && lane == 0) {
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
            // lane l loads the index of key 32 pw + l of each block, four blocks ahead
            auto ld_ent = [&](int i) -> int {
                const int ent = i * kAttnBK + pw * 32 + lane;
                return (ent < A.nsel) ? __ldg(irow + ent) : 0;
            };
            int e0 = ld_ent(0), e1 = ld_ent(1), e2 = ld_ent(2), e3 = ld_ent(3);
            for (int i = 0; i < A.nb && ok; ++i, ++rp) {
                int s_ = e0;
                if (s_ < 0 || s_ >= A.ri.n) {
                    if (i * kAttnBK + pw * 32 + lane < A.nsel) raise_error(DSA_ERR_DEVICE_DATA);
                    s_ = 0;   // any in-range row; entries past nsel are masked by the softmax
                }
                const long long myrow = PAGED ? key_row_paged(rs, r, s_) : kb + s_;
                e0 = e1; e1 = e2; e2 = e3;
                e3 = ld_ent(i + 4);
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
    } else if (warp == mma_warp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int qi = 0, gi = 0, rp = 0;
            bool ok = true;
            const uint64_t dQR = sdesc_sw64(sQR);                          // Q rope part
            // ring slot rp: keys (latent, K-major), keys (rope), values (MN-major)
            auto dK = [&](int rp_) { return sdesc_sw128(slot_addr(rp_), 16, 1024); };
            auto dR = [&](int rp_) { return sdesc_sw64(slot_addr(rp_) + 4 * C::KV_SLOT); };
            auto dV = [&](int rp_) { return sdesc_sw128(slot_addr(rp_), C::KV_SLOT, 1024); };
            // Q.K^T of block g into S buffer g & 1 (its KV item is in ring position rp_)
            auto issue_qk = [&](int g, int rp_) {
                fence_proxy_async_smem();   // rows written by cp.async, read by the tensor cores
                tc_fence_after();
                const uint32_t d = tmem_base + C::TM_S + static_cast<uint32_t>(g & 1) * kAttnBK;
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
            };
            // O += P . V of block g: P from P tile g & 1 (K-major, 128B-swizzled rows of 64 keys)
            auto issue_pv = [&](int g, int rp_, bool first) {
                const uint64_t bv = dV(rp_);
                const uint64_t bp = sdesc_sw128(sP + static_cast<uint32_t>(g & 1) * C::PT, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < kAttnBK / 16; ++kk)
                    // V (MN-major): the 4 latent slots are the 64-column chunks (LBO), 8-key groups 1 KB apart
                    tc_mma_bf16(tmem_base + C::TM_O, bp + static_cast<uint64_t>(kk * 2),
                                bv + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::IDESC_PV,
                                (!first || kk) ? 1u : 0u);
                tc_commit(pv_done(g & 1));
                tc_commit(empty(rp_ % kAttnSlots));
                // the peer's copy of block g + 2 may overwrite this rank's receive buffer g & 1:
                // this P.V has read its P half, and the factors were read before p_full
                tc_commit_multicast(pr_free(g & 1), static_cast<uint16_t>(1u << peer));
            };
            for (int r = cl; r < rows && ok; r += ncl) {
                const AttnRow A = attn_row(rs, r, k);
                if (A.nb == 0) continue;
                rp += 2;                                   // the Q item (consumed by the softmax warps)
                ok = wait_bar(q_tm_full, qi & 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const int g0 = gi, rp0 = rp, gend = gi + A.nb;
                // Q.K^T of block j needs its KV item and S buffer j & 1 free (block j-2 read by
                // every lane); P.V of block j needs both halves of its P tile.  Issue whichever is
                // ready, in block order within each kind.
                int qk_next = g0, pv_next = g0;
                uint64_t t_idle = 0;
                while (ok && pv_next < gend) {
                    bool progressed = false;
                    if (qk_next < gend) {
                        const int rq = rp0 + (qk_next - g0);
                        if (mbar_try(s_free(qk_next & 1), ((qk_next >> 1) & 1) ^ 1) &&
                            mbar_try(full(rq % kAttnSlots), (rq / kAttnSlots) & 1)) {
                            issue_qk(qk_next, rq);
                            ++qk_next;
                            progressed = true;
                        }
                    }
                    if (pv_next < qk_next && mbar_try(p_full(pv_next & 1), (pv_next >> 1) & 1) &&
                        mbar_try_cluster(pr_full(pv_next & 1), (pv_next >> 1) & 1)) {
                        tc_fence_after();
                        issue_pv(pv_next, rp0 + (pv_next - g0), pv_next == g0);
                        ++pv_next;
                        progressed = true;
                    }
                    if (progressed) {
                        t_idle = 0;
                    } else {
                        const uint64_t now = global_ns();
                        if (t_idle == 0) {
                            t_idle = now;
                        } else if (now - t_idle > timeout_ns) {
                            *s_abort = 1;
                            raise_error(DSA_ERR_TIMEOUT);
                            ok = false;
                        } else if (*s_abort) {
                            ok = false;
                        }
                    }
                }
                gi = gend;
                rp = rp0 + A.nb;
                ++qi;
            }
            tc_commit(done_bar);                          // every MMA issued has completed
            wait_bar(done_bar, 0, timeout_ns, nullptr);   // before TMEM is released
        }
    } else if (warp == copy_warp) {
        // ---------------- copy warp: sends this rank's half of each P tile to the peer ----------------
        if (lane == 0) {
            const uint32_t rP = mapa(sP, peer), rMR = mapa(sbase + C::OFF_MR, peer);
            int g = 0;
            bool ok = true;
            for (int r = cl; r < rows && ok; r += ncl) {
                const AttnRow A = attn_row(rs, r, k);
                for (int i = 0; i < A.nb && ok; ++i, ++g) {
                    const int b = g & 1;
                    // the own warps have written the rows; the peer's P.V of block g-2 has completed
                    ok = wait_bar(p_ready(b), (g >> 1) & 1, timeout_ns, s_abort) &&
                         wait_bar<true>(pr_free(b), ((g >> 1) & 1) ^ 1, timeout_ns, s_abort);
                    if (!ok) break;
                    const uint32_t rb = mapa(pr_full(b), peer);
                    const uint32_t off = static_cast<uint32_t>(b * C::PT + rank * C::PH);
                    bulk_copy_to_peer(rP + off, sP + off, C::PH, rb);
                    bulk_copy_to_peer(rMR + b * C::MB, sbase + C::OFF_MS + b * C::MB, C::MB, rb);
                    bulk_commit();
                    bulk_wait_read<0>();
                    mbar_arrive(pcopy_done(b));
                }
            }
            bulk_wait_read<0>();
        }
    } else if (warp < 4) {
        // ---------------- softmax group / Q items / epilogue (warps 0..3) ----------------
        const int h = warp * 32 + lane;              // head = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const bool own = (warp >> 1) == rank;         // this lane's head has its softmax here
        const int hl = h & 63;                        // row of the head in the 64-head exchange tiles
        int qi = 0, gi = 0, rp = 0;
        bool ok = true;
        uint32_t bulk_pending = 0;                    // this thread has issued bulk copies

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
            if (lse != nullptr && own) lse[static_cast<long long>(rr) * kAttnHeads + h] = -INFINITY;
        };
        // Rescales this lane's O row by f (warp-uniform call; f = 1 leaves it unchanged).
        auto rescale_o = [&](float f) {
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tmem_base + lane_off + C::TM_O + c0, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
                tmem_st32(tmem_base + lane_off + C::TM_O + c0, o);
            }
        };
        // the P.V of block g-2 has finished reading P tile g & 1 (and O holds it)
        auto wait_p_buffer = [&](int g) -> bool {
            if (g < 2) return true;
            return __all_sync(0xffffffffu, wait_bar(pv_done(g & 1), (((g - 2) >> 1) & 1), timeout_ns, s_abort));
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
        const uint32_t rXR = mapa(sbase + C::OFF_XR, peer);
        float l_peer = 1.f;                           // peer lanes: the denominator received last
        // Peer lanes: takes the rescale factors and denominators that came with the peer's half of
        // P tile g & 1 (block g, the i-th of the query), rescales these O rows if told to, and
        // releases the P.V of block g.  Does nothing and returns false while the peer's half has
        // not arrived, or while a rescale still has to wait for the P.V of block g - 1.
        auto try_take = [&](int g, int i) -> bool {
            const int b = g & 1;
            if (!__all_sync(0xffffffffu, mbar_test_cluster(pr_full(b), (g >> 1) & 1))) return false;
            const float* mr = reinterpret_cast<const float*>(smem + C::OFF_MR + b * C::MB);
            const float f = mr[hl];
            if (i > 0 && __any_sync(0xffffffffu, f != 1.f)) {
                // O must hold every earlier P.V before it is rescaled.  (The peer sent block g
                // after this rank's P.V of block g - 2 completed, so the phase tested is current.)
                if (!__all_sync(0xffffffffu, mbar_test(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1))) return false;
                tc_fence_after();
                rescale_o(f);
                tmem_st_wait();
            }
            l_peer = mr[64 + hl];
            tc_fence_before();
            mbar_arrive(p_full(b));
            return true;
        };
        // The output epilogue of a finished query is deferred until this lane has read S of the
        // next query's first block (and, for peer lanes, sent its partial scores): the first
        // exchange and Q.K^T of the next query then overlap the output stores.  The next query's
        // first P.V (which overwrites O) needs P from every lane, given only after the epilogue.
        int ep_r = -1, ep_gl = 0;
        float ep_l = 1.f, ep_m = 0.f;
        auto run_epilogue = [&]() -> bool {
            if (ep_r < 0) return true;
            if (!__all_sync(0xffffffffu, wait_bar(pv_done(ep_gl & 1), (ep_gl >> 1) & 1, timeout_ns, s_abort)))
                return false;
            tc_fence_after();
            const float inv = 1.f / ep_l;
            const long long orow = (static_cast<long long>(ep_r) * kAttnHeads + h) * kAttnDv + rank * 256;
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
            if (lse != nullptr && own)
                lse[static_cast<long long>(ep_r) * kAttnHeads + h] = (ep_m + log2f(ep_l)) * 0.69314718055994530942f;
            tc_fence_before();   // O has been read before the next query's first P.V overwrites it
            ep_r = -1;
            return true;
        };
        while (r < rows && ok) {
            float m = -INFINITY, l = 0.f;             // own lanes: running max and denominator
            const int g0 = gi;
            if (!own) {
                // ---- peer lanes: send this rank's partial scores of the peer's heads as soon as a
                // block's scores are in and the peer's receive buffer is free, and take the peer's
                // P whenever it has arrived.  Every condition is tested without blocking, so neither
                // stream waits behind the other and neither peer warp waits for its sibling (each
                // stages and sends its own 32 rows). ----
                const int pwi = hl >> 5;
                const uint32_t sxs = sbase + C::OFF_XS + static_cast<uint32_t>(pwi * C::XSW);
                uint8_t* xs = smem + C::OFF_XS + pwi * C::XSW + lane * 256;
                int ns = 0, nst = 0, nt = 0, nt_posted = -1;   // blocks sent, staged, taken
                uint64_t t_idle = 0;
                while (ok && nt < A.nb) {
                    bool prog = false;
                    // a staged block goes out as soon as the peer has read the previous one
                    if (nst > ns && __all_sync(0xffffffffu, mbar_test_cluster(xr_free, ((g0 + ns) & 1) ^ 1))) {
                        if (lane == 0) {
                            bulk_copy_to_peer(rXR + static_cast<uint32_t>(pwi * C::XSW), sxs, C::XSW,
                                              mapa(xr_full, peer));
                            bulk_commit();
                            bulk_pending = 1;
                        }
                        ++ns;
                        prog = true;
                        if (ns == 1) ok = run_epilogue();   // the previous query's output
                    }
                    if (ok && !prog && nt < ns) {
                        if (nt_posted != nt) {   // once per block, after the buffer's previous phase
                            if (hl == 0) mbar_expect_tx(pr_full((g0 + nt) & 1), C::P_TX);
                            nt_posted = nt;
                        }
                        if (try_take(g0 + nt, nt)) {
                            ++nt;
                            prog = true;
                        }
                    }
                    // otherwise the next block is staged once its S is in, so that only the copy
                    // waits for the peer's buffer (staging may wait for the previous copy to have
                    // read the staging buffer, so it comes after the takes)
                    if (!prog && nst == ns && nst < A.nb) {
                        const int g = g0 + nst, b = g & 1;
                        if (__all_sync(0xffffffffu, mbar_test(s_full(b), (g >> 1) & 1))) {
                            tc_fence_after();
                            uint32_t sraw[64];
                            const uint32_t ts = tmem_base + lane_off + C::TM_S + static_cast<uint32_t>(b) * kAttnBK;
                            tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(sraw));
                            tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(sraw + 32));
                            tmem_ld_wait();
                            tc_fence_before();
                            mbar_arrive(s_free(b));            // Q.K^T of block g + 2 may overwrite this buffer
                            if (lane == 0 && bulk_pending) bulk_wait_read<0>();   // the staging buffer is free
                            __syncwarp();
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                *reinterpret_cast<uint4*>(xs + (((c ^ hl) & 15) << 4)) =
                                    make_uint4(sraw[4 * c], sraw[4 * c + 1], sraw[4 * c + 2], sraw[4 * c + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            ++nst;
                            prog = true;
                        }
                    }
                    if (prog) {
                        t_idle = 0;
                    } else {
                        const uint64_t now = global_ns();
                        if (t_idle == 0) {
                            t_idle = now;
                        } else if (now - t_idle > timeout_ns) {
                            *s_abort = 1;
                            raise_error(DSA_ERR_TIMEOUT);
                            ok = false;
                        } else if (*s_abort) {
                            ok = false;
                        }
                    }
                }
            }
            for (int i = 0; i < A.nb && ok && own; ++i) {
                const int g = g0 + i, b = g & 1;
                ok = __all_sync(0xffffffffu, wait_bar(s_full(b), (g >> 1) & 1, timeout_ns, s_abort));
                if (!ok) break;
                tc_fence_after();
                uint32_t sraw[64];
                const uint32_t ts = tmem_base + lane_off + C::TM_S + static_cast<uint32_t>(b) * kAttnBK;
                tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(sraw));
                tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(sraw + 32));
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(s_free(b));                // Q.K^T of block g + 2 may overwrite this buffer
                {
                    // ---- own lanes: complete the scores, softmax, write P for both ranks ----
                    if (i == 0) {
                        ok = run_epilogue();           // the previous query's output
                        if (!ok) break;
                    }
                    // this rank's half of P tile b and factor buffer b are free once the P.V of block
                    // g-2 has completed here and their copy to the peer has been read
                    ok = wait_p_buffer(g) &&
                         __all_sync(0xffffffffu, wait_bar(pcopy_done(b), ((g >> 1) & 1) ^ 1, timeout_ns, s_abort));
                    if (!ok) break;
                    if (hl == 0) mbar_expect_tx(xr_full, C::XB);
                    ok = __all_sync(0xffffffffu, wait_bar<true>(xr_full, g & 1, timeout_ns, s_abort));
                    if (!ok) break;
                    float sv[64];
                    const uint8_t* xr = smem + C::OFF_XR + hl * 256;
                    uint32_t dep = 0;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float4 v = *reinterpret_cast<const float4*>(xr + (((c ^ hl) & 15) << 4));
                        dep |= __float_as_uint(v.x);
                        sv[4 * c + 0] = __uint_as_float(sraw[4 * c + 0]) + v.x;
                        sv[4 * c + 1] = __uint_as_float(sraw[4 * c + 1]) + v.y;
                        sv[4 * c + 2] = __uint_as_float(sraw[4 * c + 2]) + v.z;
                        sv[4 * c + 3] = __uint_as_float(sraw[4 * c + 3]) + v.w;
                    }
                    // Hand XR back to the peer, whose next bulk copy overwrites it, once this
                    // warp's loads of it have returned (a zeroing step the compiler could fold
                    // let the arrive overtake them, and the peer overwrite the first rows).
                    if (lane == 0) mbar_arrive_cluster_after(mapa(xr_free, peer), dep, opaque_zero);
                    // columns past the last valid entry are masked (identical for every head)
                    const int nvalid = A.nsel - i * kAttnBK;
                    if (nvalid < kAttnBK) {
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (j >= nvalid) sv[j] = -INFINITY;
                    }
                    // With a positive scale the row maximum is taken on the raw scores and the
                    // scale is folded into the exponent's FMA (one instruction per score).
                    const bool pos_scale = scale_log2 > 0.f;
                    float mx = -INFINITY;
                    if (pos_scale) {
                        float t8[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) t8[q] = sv[q];
#pragma unroll
                        for (int j = 8; j < 64; ++j) t8[j & 7] = fmaxf(t8[j & 7], sv[j]);
                        mx = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                                   fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
                        mx *= scale_log2;
                    } else {
#pragma unroll
                        for (int j = 0; j < 64; ++j) {
                            sv[j] = (j < nvalid) ? sv[j] * scale_log2 : -INFINITY;
                            mx = fmaxf(mx, sv[j]);
                        }
                    }
                    const float m_new = fmaxf(m, mx);
                    const bool resc = m_new > m + 8.f;       // lazy rescale (always true on the first block)
                    float factor = resc ? fast_exp2(m - m_new) : 1.f;
                    if (i == 0) factor = 1.f;                // the first P.V overwrites O
                    if (resc) {
                        l *= factor;
                        m = m_new;
                    }
                    // P = 2^(z - m) in bf16 (pairs of keys per 32-bit column); l sums the fp32 values
                    // before rounding, in four independent partial sums
                    const float zs = pos_scale ? scale_log2 : 1.f;
                    uint32_t pk[32];
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = fast_exp2(fmaf(sv[2 * j], zs, -m)), p1 = fast_exp2(fmaf(sv[2 * j + 1], zs, -m));
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(p0, p1);
                        ls[j & 3] += p0 + p1;
                        pk[j] = *reinterpret_cast<const uint32_t*>(&pr);
                    }
                    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    uint8_t* pt = smem + C::OFF_P + b * C::PT + h * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(pt + (((c ^ h) & 7) << 4)) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    float* ms = reinterpret_cast<float*>(smem + C::OFF_MS + b * C::MB);
                    ms[hl] = factor;
                    ms[64 + hl] = l;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_ready(b));   // the copy warp sends these rows to the peer
                    if (i > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
                        ok = __all_sync(0xffffffffu,
                                        wait_bar(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1, timeout_ns, s_abort));
                        if (!ok) break;
                        tc_fence_after();
                        rescale_o(factor);
                        tmem_st_wait();
                    }
                    tc_fence_before();
                    mbar_arrive(p_full(b));
                }
            }
            if (!ok) break;
            gi = g0 + A.nb;
            rp += A.nb;
            const int r_cur = r;
            const float l_fin = own ? l : l_peer;
            const float m_fin = m;
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
            // ---------------- epilogue of the finished query: deferred (see run_epilogue) ----------------
            ep_r = r_cur;
            ep_gl = gi - 1;
            ep_l = l_fin;
            ep_m = m_fin;
            if (!ok) break;
        }
        if (ok) ok = run_epilogue();                  // the last query's output
        if (bulk_pending) bulk_wait_read<0>();
        (void)qi;
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();             // the peer no longer writes into this CTA's shared memory
    if (warp == mma_warp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace dsa
