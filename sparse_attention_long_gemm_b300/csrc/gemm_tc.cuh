// gemm_tc.cuh -- the Lightning Indexer's input projections on the sm_103a
// tensor cores, and the decode step's key-cache append.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the indexer scores
// queries taken from the MLA query latent through its projection wq_b (sized
// by q_lora_rank), weights its heads with the weights_proj module, and keeps
// its own single-head key cache of index_head_dim per token, updated through
// update_indexer().  The projections are bias-free linear maps,
//     C[M, N] = A[M, K] . B[N, K]^T
// with A the activations (tokens x K) and B the weight (N outputs x K), both
// bf16 with K contiguous; the products accumulate in fp32 in tensor memory and
// C is written as bf16 (indexer queries and keys) or fp32 (head weights).
//
// gemm_tc_kernel: persistent, 128 x BN tiles of C (192 threads per CTA; as
// many CTAs as fit on the SMs at once: one for BN = 256 and 128, two for 64).
//   - one thread streams 128 x 64 tiles of A and BN x 64 tiles of B by TMA
//     (128-byte swizzle) through a 4-stage ring;
//   - one thread issues tcgen05.mma kind::f16 (M = 128, N = BN, K = 16, four
//     per 64-wide K step) into one of two BN-column fp32 accumulators in
//     tensor memory and frees each stage with tcgen05.commit;
//   - four epilogue warps read a finished accumulator's lanes (rows) back with
//     tcgen05.ld and store them, converted, with 16-byte stores, while the
//     next tile accumulates into the other half.
// Rows past M and columns past N are zero-filled by TMA on load and masked on
// store; a K that is not a multiple of 64 reads zeros past its end.
//
// update_indexer_kernel: one CTA per sequence copies the new token's indexer
// key and latent row to position cache_seqlens[b] of its caches (dense, or
// paged through a block table) and advances the length.  A length outside
// [0, max_ctx) (no room) or a page outside the pool writes nothing and raises
// DSA_ERR_DEVICE_DATA.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "rows.cuh"

namespace dsa {

constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;   // warp 0: TMA, warp 1: tensor memory and MMA, warps 2..5: epilogue

template <int BN>
struct GemmTc {
    static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
    static constexpr int A_BYTES = kGemmBM * kGemmBK * 2;      // 16 KB
    static constexpr int B_BYTES = BN * kGemmBK * 2;           // 8 .. 32 KB
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int OFF_BAR = kGemmStages * STAGE;
    static constexpr int NBAR = 2 * kGemmStages + 5;           // full[S], empty[S], acc_full[2], acc_empty[2], done
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;          // + alignment slack
    static constexpr uint32_t IDESC = idesc_bf16(kGemmBM, BN, false, false);
    static constexpr int TMEM_COLS = 2 * BN;                   // two accumulators
};
static_assert(GemmTc<256>::SMEM <= 232448, "gemm shared memory exceeds the per-CTA limit");
static_assert(GemmTc<64>::STAGE % 1024 == 0 && GemmTc<128>::STAGE % 1024 == 0 && GemmTc<256>::STAGE % 1024 == 0,
              "stages hold 128B-swizzled tiles (1024-byte atoms)");

// Persistent: CTA b takes tiles b, b + gridDim.x, ... of the (M / 128) x (N / BN) grid, N fastest
// (neighbouring CTAs share the A rows in L2).  The accumulator alternates between two halves of
// tensor memory, so the epilogue of one tile overlaps the MMAs of the next.
template <int BN, bool OUT_BF16>
__global__ void __launch_bounds__(kGemmThreads)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, int M, int N,
               int K, void* __restrict__ c, long long ldc, unsigned long long timeout_ns) {
    using G = GemmTc<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + G::OFF_BAR;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kGemmStages + s); };
    auto acc_full = [&](int a) { return bar0 + 8u * (2 * kGemmStages + a); };
    auto acc_empty = [&](int a) { return bar0 + 8u * (2 * kGemmStages + 2 + a); };
    const uint32_t done_bar = bar0 + 8u * (2 * kGemmStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + G::OFF_MISC + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = (K + kGemmBK - 1) / kGemmBK;
    const int tiles_n = (N + BN - 1) / BN;
    const int ntiles = tiles_n * ((M + kGemmBM - 1) / kGemmBM);

    if (tid == 0) {
        for (int s = 0; s < kGemmStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(acc_full(a), 1); mbar_init(acc_empty(a), 128); }
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int n0 = (t % tiles_n) * BN, m0 = (t / tiles_n) * kGemmBM;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % kGemmStages;
                    ok = wait_bar(empty(s), ((it / kGemmStages) & 1) ^ 1, timeout_ns, s_abort);
                    if (!ok) break;
                    const uint32_t st = sbase + static_cast<uint32_t>(s * G::STAGE);
                    mbar_expect_tx(full(s), G::STAGE);
                    tma_load_2d(st, &tm_a, kb * kGemmBK, m0, full(s));
                    tma_load_2d(st + G::A_BYTES, &tm_b, kb * kGemmBK, n0, full(s));
                }
            }
            if (!ok) sleep_ns(1000000ull);   // loads already issued land before the CTA exits
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, ti = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++ti) {
                const int a = ti & 1;
                // the epilogue has read this accumulator's previous tile
                ok = wait_bar(acc_empty(a), ((ti >> 1) & 1) ^ 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(a * BN);
                for (int kb = 0; kb < nk && ok; ++kb, ++it) {
                    const int s = it % kGemmStages;
                    ok = wait_bar(full(s), (it / kGemmStages) & 1, timeout_ns, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t st = sbase + static_cast<uint32_t>(s * G::STAGE);
                    const uint64_t da = sdesc_sw128(st, 16, 1024), db = sdesc_sw128(st + G::A_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk)
                        tc_mma_bf16(d, da + static_cast<uint64_t>((kk * 32) >> 4),
                                    db + static_cast<uint64_t>((kk * 32) >> 4), G::IDESC, (kb | kk) ? 1u : 0u);
                    tc_commit(empty(s));
                }
                if (ok) tc_commit(acc_full(a));
            }
            tc_commit(done_bar);                          // every MMA issued has completed
            wait_bar(done_bar, 0, timeout_ns, nullptr);   // before tensor memory is released
        }
    } else {
        // ---------------- epilogue: warp w reads accumulator lanes (rows) 32 (w % 4) .. +31 ----------------
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        int ti = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++ti) {
            const int a = ti & 1;
            ok = __all_sync(0xffffffffu, wait_bar(acc_full(a), (ti >> 1) & 1, timeout_ns, s_abort));
            if (!ok) break;
            tc_fence_after();
            const int n0 = (t % tiles_n) * BN, m0 = (t / tiles_n) * kGemmBM;
            const int row = m0 + quad * 32 + lane;
            const uint32_t taddr = tmem + lane_off + static_cast<uint32_t>(a * BN);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(taddr + static_cast<uint32_t>(c0), v);
                tmem_ld_wait();
                const int col = n0 + c0;
                if (row >= M || col >= N) continue;
                const bool whole = col + 32 <= N;
                if constexpr (OUT_BF16) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(c) + static_cast<long long>(row) * ldc + col;
                    if (whole) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t pk[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[8 * q + 2 * e]),
                                                                               __uint_as_float(v[8 * q + 2 * e + 1]));
                                pk[e] = *reinterpret_cast<const uint32_t*>(&h);
                            }
                            reinterpret_cast<uint4*>(dst)[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < N - col) dst[j] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                } else {
                    float* dst = static_cast<float*>(c) + static_cast<long long>(row) * ldc + col;
                    if (whole) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            reinterpret_cast<float4*>(dst)[q] =
                                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < N - col) dst[j] = __uint_as_float(v[j]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acc_empty(a));   // the MMA thread may start the tile after next in this half
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, G::TMEM_COLS);
    }
}

constexpr int kUpdThreads = 128;

// One CTA per sequence: the new token's indexer key (k_bytes per sequence) and latent row
// (kv_bytes) go to the row of position cache_seqlens[b] in idx_cache and kv_cache (dense
// [batch, max_ctx, .] caches, or page pools through the block table of `rs`), and the length
// grows by one.  Row sizes are multiples of 16 bytes and the arrays 16-byte aligned.
__global__ void __launch_bounds__(kUpdThreads)
update_indexer_kernel(RowSpec rs, const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ kv_new,
                      int k_bytes, int kv_bytes, int* __restrict__ cache_seqlens, uint8_t* __restrict__ idx_cache,
                      uint8_t* __restrict__ kv_cache) {
    const int b = blockIdx.x;
    if (b >= rs.batch) return;
    const int p = cache_seqlens[b];
    bool ok = p >= 0 && p < rs.max_len;   // else no room (or a corrupt length)
    long long slot = static_cast<long long>(b) * rs.max_len + p;
    if (ok && rs.pages != nullptr) {
        // a page outside the pool is reported and nothing is written (the readers' fallback to
        // page 0 would overwrite another sequence's rows here)
        const int pg = __ldg(rs.pages + static_cast<long long>(b) * rs.max_pages + (p >> rs.page_log2));
        ok = pg >= 0 && pg < rs.num_pages;
        slot = (static_cast<long long>(pg) << rs.page_log2) + (p & ((1 << rs.page_log2) - 1));
    }
    if (!ok) {
        if (threadIdx.x == 0) raise_error(DSA_ERR_DEVICE_DATA);
        return;
    }
    const uint4* ks = reinterpret_cast<const uint4*>(k_new + static_cast<long long>(b) * k_bytes);
    uint4* kd = reinterpret_cast<uint4*>(idx_cache + slot * k_bytes);
    for (int i = threadIdx.x; i < k_bytes / 16; i += kUpdThreads) kd[i] = ks[i];
    const uint4* vs = reinterpret_cast<const uint4*>(kv_new + static_cast<long long>(b) * kv_bytes);
    uint4* vd = reinterpret_cast<uint4*>(kv_cache + slot * kv_bytes);
    for (int i = threadIdx.x; i < kv_bytes / 16; i += kUpdThreads) vd[i] = vs[i];
    __syncthreads();   // every thread has read the length before it changes
    if (threadIdx.x == 0) cache_seqlens[b] = p + 1;
}

}  // namespace dsa
