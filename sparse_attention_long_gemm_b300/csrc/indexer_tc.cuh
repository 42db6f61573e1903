// indexer_tc.cuh -- Lightning Indexer on the sm_103a tensor cores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", Lightning Indexer,
// at the DeepseekV32Config sizes index_n_heads = 64, index_head_dim = 128:
//     I[t,s] = sum_j w[t,j] * max(0, q_I[t,j,:] . k_I[s,:])   for s <= t.
//
// The contraction is computed transposed, S^T = k_I . q_I^T: a tile of 128
// keys is the MMA's M (one TMEM lane per key) and NQ queries x 64 heads its
// N, K = 128.  Each epilogue thread then owns one key and sums its 64 heads
// for each query in registers (ReLU and the w-weighted head sum fused), so
// the per-head scores never leave TMEM and no cross-lane reduction is
// needed.  Only the causal part (s <= t) is computed and written.
//
// Warp roles (64 + 128 NQ threads, one CTA per SM, persistent over work units):
//   warp 0      TMA producer: query block (NQ*64 rows x 128, once per unit)
//               and key tiles (128 x 128) into 128B-swizzled shared memory;
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread);
//   warps 2..   epilogue: per TMEM lane quadrant, two warps for the 4-query
//               bf16 prefill block (two queries each), four for the FP8 form
//               (one query each), one in decode; a warp's queries' accumulator
//               columns are loaded before one wait, and each 64-head sum runs
//               as packed pairs in independent partial sums.
// Two TMEM accumulators alternate so the epilogue of one key tile overlaps
// the MMAs of the next.
//
// Work unit = (query block of NQ consecutive queries of one sequence, a run
// of at most `kc` key tiles).  Bounding the run length keeps every unit
// about the same size, so a static round-robin over CTAs balances the
// causal triangle (and, in decode, long caches) without sorting.
#pragma once

#include <cuda.h>

#include "rows.cuh"

namespace dsa {

constexpr int kIdxHeads = 64;
constexpr int kIdxDim = 128;
constexpr int kIdxTileKeys = 128;
constexpr int kIdxRoleThreads = 64;      // warp 0 TMA producer, warp 1 MMA issuer
constexpr int kIdxTcMaxBatch = 256;      // sequences per launch (the host splits longer batches)

// Packed fp32 pairs (sm_100 family): d = a * b + c on both halves at once.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t x, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// F8: operands are E4M3 codes (one byte per element, so a 128-d row is one 128-byte swizzled
// row and each MMA takes K = 32) instead of bf16 (two 128-byte halves per row, K = 16).
template <int NQ, int KSTAGES, int QBUF, bool F8 = false>
struct IdxTc {
    static constexpr int ESZ = F8 ? 1 : 2;                    // bytes per element
    static constexpr int KH = F8 ? 1 : 2;                     // 128-byte parts of a 128-d row
    static constexpr int BN = NQ * kIdxHeads;                 // MMA N
    // epilogue warps: one per TMEM lane quadrant and query of the block for the FP8 form, whose
    // MMAs take half the time so that the epilogue must keep pace with twice the tiles; two
    // per quadrant (two queries each) for the bf16 prefill block, one per quadrant in decode.
    // (Each sub-partition's 16 Ki registers hold a quarter of the warps: 10 warps allow 168
    // registers a thread, 18 allow 96.)
    static constexpr int EPI_WARPS = F8 ? 4 * NQ : (NQ > 1 ? 2 * NQ : 4);
    static constexpr int QPW = NQ * 4 / EPI_WARPS;            // queries per epilogue warp
    static constexpr int THREADS = kIdxRoleThreads + 32 * EPI_WARPS;
    static constexpr int Q_BYTES = BN * kIdxDim * ESZ;        // one query block
    static constexpr int Q_HALF = BN * 128;                   // one 128-byte part of it
    static constexpr int K_BYTES = kIdxTileKeys * kIdxDim * ESZ;
    static constexpr int K_HALF = kIdxTileKeys * 128;
    static constexpr int TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
    static constexpr int OFF_K = QBUF * Q_BYTES;
    static constexpr int OFF_BAR = OFF_K + KSTAGES * K_BYTES;
    static constexpr int NBAR = 2 * QBUF + 2 * KSTAGES + 4 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_TABLE = OFF_MISC + 16;
    static constexpr int SMEM = OFF_TABLE + (kIdxTcMaxBatch + 1) * 4 + 1024;  // + alignment slack
    static constexpr uint32_t IDESC = F8 ? idesc_e4m3(128, BN) : idesc_bf16(128, BN, false, false);
};

struct IdxUnit {
    int q_row0;          // global row of the block's first query
    int nq;              // valid queries in the block (1..NQ)
    int t0;              // sequence position of the first query
    long long key_base;  // key-tensor row of position 0
    int kt0, kt1;        // key tiles [kt0, kt1)
};

// number of chunks of key tiles for a query block in causal band m
__device__ __forceinline__ int idx_chunks(int m, int kc) { return (m + kc) / kc; }   // ceil((m+1)/kc)
// sum over bands m' < M of idx_chunks(m')
__device__ __forceinline__ long long idx_chunks_below(int M, int kc) {
    const long long a = M / kc, rr = M % kc;
    return kc * a * (a + 1) / 2 + rr * (a + 1);
}

template <int NQ>
struct IdxSched {
    static constexpr int QPB = kIdxTileKeys / NQ;   // query blocks per band of 128 positions

    // units before query block q of a sequence
    __device__ __forceinline__ static long long units_before(int q, int kc) {
        const int band = q / QPB;
        return QPB * idx_chunks_below(band, kc) + static_cast<long long>(q - band * QPB) * idx_chunks(band, kc);
    }
    // units of sequence b (0 when its length is invalid)
    __device__ static long long seq_units(const RowSpec& rs, int b, int kc) {
        if (rs.decode) {
            const int n = __ldg(rs.lens + b);
            if (n < 1 || n > rs.max_len) { raise_error(DSA_ERR_DEVICE_DATA); return 0; }
            const int ntiles = (n + kIdxTileKeys - 1) / kIdxTileKeys;
            return (ntiles + kc - 1) / kc;
        }
        const int lo = __ldg(rs.lens + b), hi = __ldg(rs.lens + b + 1);
        const int len = hi - lo;
        if (lo < 0 || len < 0 || len > rs.max_len) { raise_error(DSA_ERR_DEVICE_DATA); return 0; }
        const int nqb = (len + NQ - 1) / NQ;
        return units_before(nqb, kc);
    }
    // unit v of sequence b
    __device__ static IdxUnit unit(const RowSpec& rs, int b, long long v, int kc) {
        IdxUnit U;
        if (rs.decode) {
            const int n = __ldg(rs.lens + b);
            const int ntiles = (n + kIdxTileKeys - 1) / kIdxTileKeys;
            U.q_row0 = rs.base + b;
            U.nq = 1;
            U.t0 = n - 1;
            U.key_base = static_cast<long long>(rs.base + b) * rs.max_len;
            U.kt0 = static_cast<int>(v) * kc;
            U.kt1 = min(U.kt0 + kc, ntiles);
            return U;
        }
        const int lo = __ldg(rs.lens + b), len = __ldg(rs.lens + b + 1) - lo;
        const int nqb = (len + NQ - 1) / NQ;
        int ql = 0, qh = nqb - 1;   // largest q with units_before(q) <= v
        while (ql < qh) {
            const int mid = (ql + qh + 1) >> 1;
            if (units_before(mid, kc) <= v) ql = mid; else qh = mid - 1;
        }
        const int c = static_cast<int>(v - units_before(ql, kc));
        const int band = ql / QPB;
        U.t0 = ql * NQ;
        U.nq = min(NQ, len - U.t0);
        U.q_row0 = lo + U.t0;
        U.key_base = lo;
        U.kt0 = c * kc;
        U.kt1 = min(U.kt0 + kc, band + 1);
        return U;
    }
};

// F8: q / k are E4M3 codes of the rotated vectors, w holds w * s_q (the query scales folded
// in) and ksc the key scales s_k, applied per key after the head sum (both scales are positive,
// so they commute with the ReLU).
template <int NQ, int KSTAGES, int QBUF, bool F8 = false, bool PAGED = false>
__global__ void __launch_bounds__(IdxTc<NQ, KSTAGES, QBUF, F8>::THREADS, 1)
indexer_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, RowSpec rs,
                  const float* __restrict__ w, const float* __restrict__ ksc, float* __restrict__ scores,
                  long long ld, int kc, unsigned long long timeout_ns) {
    using C = IdxTc<NQ, KSTAGES, QBUF, F8>;
    using Sch = IdxSched<NQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase, sK = sbase + C::OFF_K;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto q_full = [&](int i) { return bar0 + 8u * i; };
    auto q_empty = [&](int i) { return bar0 + 8u * (QBUF + i); };
    auto k_full = [&](int i) { return bar0 + 8u * (2 * QBUF + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (2 * QBUF + KSTAGES + i); };
    auto acc_full = [&](int i) { return bar0 + 8u * (2 * QBUF + 2 * KSTAGES + i); };
    auto acc_empty = [&](int i) { return bar0 + 8u * (2 * QBUF + 2 * KSTAGES + 2 + i); };
    const uint32_t done_bar = bar0 + 8u * (2 * QBUF + 2 * KSTAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* s_pref = reinterpret_cast<int*>(smem + C::OFF_TABLE);   // units before sequence b

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < QBUF; ++i) { mbar_init(q_full(i), 1); mbar_init(q_empty(i), 1); }
        for (int i = 0; i < KSTAGES; ++i) { mbar_init(k_full(i), 1); mbar_init(k_empty(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(acc_full(i), 1); mbar_init(acc_empty(i), 32 * C::EPI_WARPS); }
        mbar_init(done_bar, 1);
        *s_abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // per-sequence unit prefix (serial; the batch is small on this path)
    if (tid == 32 * 2) {
        long long acc = 0;
        for (int b = 0; b < rs.batch; ++b) {
            s_pref[b] = static_cast<int>(acc);
            acc += Sch::seq_units(rs, b, kc);
        }
        s_pref[rs.batch] = static_cast<int>(acc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total_units = s_pref[rs.batch];

    auto get_unit = [&](int u) {
        int bl = 0, bh = rs.batch - 1;
        while (bl < bh) {
            const int mid = (bl + bh + 1) >> 1;
            if (s_pref[mid] <= u) bl = mid; else bh = mid - 1;
        }
        return Sch::unit(rs, bl, u - s_pref[bl], kc);
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer ----------------
        int it_q = 0, it_k = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            const IdxUnit U = get_unit(u);
            const int qb = it_q % QBUF;
            ok = wait_bar(q_empty(qb), ((it_q / QBUF) & 1) ^ 1, timeout_ns, s_abort);
            if (!ok) break;
            mbar_expect_tx(q_full(qb), C::Q_BYTES);
            for (int kh = 0; kh < C::KH; ++kh)
                tma_load_2d(sQ + qb * C::Q_BYTES + kh * C::Q_HALF, &tm_q, kh * 64, U.q_row0 * kIdxHeads, q_full(qb));
            for (int kt = U.kt0; kt < U.kt1; ++kt) {
                const int s = it_k % KSTAGES;
                ok = wait_bar(k_empty(s), ((it_k / KSTAGES) & 1) ^ 1, timeout_ns, s_abort);
                if (!ok) break;
                mbar_expect_tx(k_full(s), C::K_BYTES);
                const int krow = static_cast<int>(PAGED ? key_row_paged(rs, U.q_row0, kt * kIdxTileKeys)
                                                        : U.key_base + static_cast<long long>(kt) * kIdxTileKeys);
                for (int kh = 0; kh < C::KH; ++kh)
                    tma_load_2d(sK + s * C::K_BYTES + kh * C::K_HALF, &tm_k, kh * 64, krow, k_full(s));
                ++it_k;
            }
            ++it_q;
        }
        if (!ok) sleep_ns(2000000ull);  // let copies already issued land before the CTA exits
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer ----------------
        int it_q = 0, it_k = 0, it_acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            const IdxUnit U = get_unit(u);
            const int qb = it_q % QBUF;
            ok = wait_bar(q_full(qb), (it_q / QBUF) & 1, timeout_ns, s_abort);
            if (!ok) break;
            tc_fence_after();
            for (int kt = U.kt0; kt < U.kt1; ++kt) {
                const int s = it_k % KSTAGES;
                const int ab = it_acc & 1;
                ok = wait_bar(k_full(s), (it_k / KSTAGES) & 1, timeout_ns, s_abort) &&
                     wait_bar(acc_empty(ab), ((it_acc >> 1) & 1) ^ 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(ab * C::BN);
#pragma unroll
                for (int kh = 0; kh < C::KH; ++kh) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {   // 32 bytes of K per MMA: 16 bf16 or 32 E4M3
                        const uint64_t a = sdesc_sw128(sK + s * C::K_BYTES + kh * C::K_HALF + kk * 32, 16, 1024);
                        const uint64_t b = sdesc_sw128(sQ + qb * C::Q_BYTES + kh * C::Q_HALF + kk * 32, 16, 1024);
                        if constexpr (F8) tc_mma_e4m3(d, a, b, C::IDESC, (kh | kk) ? 1u : 0u);
                        else tc_mma_bf16(d, a, b, C::IDESC, (kh | kk) ? 1u : 0u);
                    }
                }
                tc_commit(k_empty(s));
                tc_commit(acc_full(ab));
                ++it_k;
                ++it_acc;
            }
            if (!ok) break;
            tc_commit(q_empty(qb));
            ++it_q;
        }
        tc_commit(done_bar);                       // every MMA issued has completed
        wait_bar(done_bar, 0, timeout_ns, nullptr);  // before TMEM is released
    } else if (warp >= 2) {
        // ---------------- epilogue ----------------
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;          // which group of the block's queries this warp takes
        constexpr int QPH = C::QPW;                // queries per warp
        const int row = quad * 32 + lane;          // key within the tile = TMEM lane
        int it_acc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            const IdxUnit U = get_unit(u);
            for (int kt = U.kt0; kt < U.kt1; ++kt) {
                const int ab = it_acc & 1;
                ok = wait_bar(acc_full(ab), (it_acc >> 1) & 1, timeout_ns, s_abort);
                if (!ok) break;
                tc_fence_after();
                const int s = kt * kIdxTileKeys + row;
                const int q0 = half * QPH;
                float sk = 0.f;   // F8: this key's scale (keys past the causal range are never written)
                if constexpr (F8) {
                    if (s <= U.t0 + U.nq - 1)
                        sk = __ldg(ksc + (PAGED ? key_row_paged(rs, U.q_row0, s) : U.key_base + s));
                }
                (void)sk;
                if (q0 < U.nq) {   // warp-uniform
                    uint32_t v[QPH][64];
#pragma unroll
                    for (int qq = 0; qq < QPH; ++qq) {
                        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                               static_cast<uint32_t>(ab * C::BN + (q0 + qq) * kIdxHeads);
                        tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(v[qq]));
                        tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(v[qq] + 32));
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int qq = 0; qq < QPH; ++qq) {
                        const int qi = q0 + qq;
                        if (qi >= U.nq) break;     // warp-uniform
                        const float4* w4 = reinterpret_cast<const float4*>(w + static_cast<long long>(U.q_row0 + qi) * kIdxHeads);
                        // ReLU per head, then the w-weighted sum as packed fp32x2 FMAs (two heads per
                        // instruction), in two independent pairs of partial sums
                        uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
                        for (int j4 = 0; j4 < 16; ++j4) {
                            const float4 ww = __ldg(w4 + j4);
                            const uint64_t wa = pack_f32x2(ww.x, ww.y), wb = pack_f32x2(ww.z, ww.w);
                            const uint64_t va = pack_f32x2(fmaxf(__uint_as_float(v[qq][4 * j4 + 0]), 0.f),
                                                           fmaxf(__uint_as_float(v[qq][4 * j4 + 1]), 0.f));
                            const uint64_t vb = pack_f32x2(fmaxf(__uint_as_float(v[qq][4 * j4 + 2]), 0.f),
                                                           fmaxf(__uint_as_float(v[qq][4 * j4 + 3]), 0.f));
                            acc2[0] = fma_f32x2(wa, va, acc2[0]);
                            acc2[1] = fma_f32x2(wb, vb, acc2[1]);
                        }
                        float acc[4];
                        unpack_f32x2(acc2[0], acc[0], acc[1]);
                        unpack_f32x2(acc2[1], acc[2], acc[3]);
                        float val = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                        if constexpr (F8) val *= sk;
                        if (s <= U.t0 + qi) scores[static_cast<long long>(U.q_row0 + qi) * ld + s] = val;
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty(ab));
                ++it_acc;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace dsa
