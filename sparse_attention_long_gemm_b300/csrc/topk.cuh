// topk.cuh -- per-query top-k selection by radix select over fp32 scores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", fine-grained token
// selection: keep the index_topk highest-scoring positions of each query
// (all of them when there are at most index_topk).  Equal scores go to the
// lower position.  Output: ascending positions, -1 padded.
//
// One CTA (1024 threads) per row.  Scores become order-preserving 32-bit
// keys (score_key).  Three histogram passes over 11 + 11 + 10 key bits
// find the exact key T of the k-th largest score and how many of the
// scores equal to T must be kept ("need"); a final pass in position order
// keeps every key > T and the first `need` keys == T, computing output
// slots with a block-wide prefix sum, so the result is sorted by position
// and does not depend on thread timing.  Pass 1 reads the row from HBM; the
// later passes find it in L2.
#pragma once

#include "rows.cuh"

namespace dsa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

// Exclusive prefix sum over the block (all kTopkThreads threads call it).
// Returns this thread's exclusive prefix; *total gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
        uint32_t t = (lane < kTopkWarps) ? s_warp[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kTopkWarps) s_warp[lane] = t;   // inclusive warp totals
    }
    __syncthreads();
    const uint32_t warp_excl = (wid == 0) ? 0u : s_warp[wid - 1];
    *total = s_warp[kTopkWarps - 1];
    __syncthreads();   // s_warp may be reused by the caller's next scan
    return warp_excl + x - v;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(RowSpec rs, const float* __restrict__ scores, long long ld, int k, int* __restrict__ idx_out) {
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t s_warp[kTopkWarps];
    __shared__ uint32_t s_digit, s_above;

    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    int* out = idx_out + static_cast<long long>(r) * k;
    const RowInfo ri = row_info(rs, r);
    const int n = ri.ok ? ri.n : 0;
    if (n <= k) {  // every candidate is kept (or the row is invalid: all -1)
        for (int i = tid; i < k; i += kTopkThreads) out[i] = (i < n) ? i : -1;
        return;
    }
    const float* row = scores + static_cast<long long>(r) * ld;
    const float4* row4 = reinterpret_cast<const float4*>(row);
    const int n4 = (n + 3) >> 2;

    uint32_t prefix = 0;
    uint32_t need = static_cast<uint32_t>(k);
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = (pass == 0) ? 21 : (pass == 1 ? 10 : 0);
        const int bits = (pass == 2) ? 10 : 11;
        const int nb = 1 << bits;
        const uint32_t mask = static_cast<uint32_t>(nb - 1);
        const int hi_shift = shift + bits;
        for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        for (int i4 = tid; i4 < n4; i4 += kTopkThreads) {
            const float4 v = __ldg(row4 + i4);
            const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (i4 * 4 + e < n) {
                    const uint32_t key = score_key(vals[e]);
                    if (pass == 0 || (key >> hi_shift) == prefix) atomicAdd(&hist[(key >> shift) & mask], 1u);
                }
            }
        }
        __syncthreads();
        // thread t owns bins (from the top) nb-1-t*per .. nb-per-t*per
        const int per = nb / kTopkThreads;   // 2 or 1
        uint32_t cnt[2] = {0u, 0u};
        for (int e = 0; e < per; ++e) cnt[e] = hist[nb - 1 - tid * per - e];
        uint32_t tot;
        const uint32_t above0 = block_excl_scan(cnt[0] + cnt[1], s_warp, &tot);
        uint32_t above = above0;
        for (int e = 0; e < per; ++e) {
            if (above < need && need <= above + cnt[e]) {
                s_digit = static_cast<uint32_t>(nb - 1 - tid * per - e);
                s_above = above;
            }
            above += cnt[e];
        }
        __syncthreads();
        prefix = (prefix << bits) | s_digit;
        need -= s_above;
        __syncthreads();
    }
    const uint32_t T = prefix;

    // emit, in position order, keys > T and the first `need` keys == T
    uint32_t eq_seen = 0, sel_seen = 0;
    for (int base4 = 0; base4 < n4; base4 += kTopkThreads) {
        const int i4 = base4 + tid;
        uint32_t kk[4] = {0u, 0u, 0u, 0u};
        bool in[4] = {false, false, false, false};
        if (i4 < n4) {
            const float4 v = __ldg(row4 + i4);
            const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                in[e] = (i4 * 4 + e < n);
                kk[e] = score_key(vals[e]);
            }
        }
        uint32_t c_gt = 0, c_eq = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            c_gt += (in[e] && kk[e] > T) ? 1u : 0u;
            c_eq += (in[e] && kk[e] == T) ? 1u : 0u;
        }
        uint32_t tot;
        const uint32_t pre = block_excl_scan(c_gt | (c_eq << 16), s_warp, &tot);
        const uint32_t gt_before = pre & 0xffffu, eq_before = pre >> 16;
        const uint32_t gt_tot = tot & 0xffffu, eq_tot = tot >> 16;
        const uint32_t rem = (need > eq_seen) ? need - eq_seen : 0u;   // equal keys still to keep
        uint32_t slot = sel_seen + gt_before + min(eq_before, rem);
        uint32_t eq_i = eq_before;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (!in[e]) continue;
            bool take = kk[e] > T;
            if (kk[e] == T) {
                take = eq_i < rem;
                ++eq_i;
            }
            if (take) out[slot++] = i4 * 4 + e;
        }
        sel_seen += gt_tot + min(eq_tot, rem);
        eq_seen += eq_tot;
    }
}

}  // namespace dsa
