// topk.cuh -- per-query top-k selection by radix select over fp32 scores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", fine-grained token
// selection: keep the index_topk highest-scoring positions of each query
// (all of them when there are at most index_topk).  Equal scores go to the
// lower position.  Output: ascending positions, -1 padded.
//
// topk_smem_kernel (rows of at most kTopkSmemKeys positions): persistent CTAs
// of 1024 threads, one row at a time, each row read from HBM ONCE (prefetched
// into L2 while the CTA works on its previous row) with its keys kept in
// shared memory.  After the first histogram, the positions whose top key bits
// reach the k-th largest key's bin are listed in position order; the two
// refining radix passes and the ordered emit then run over that short list.
// Rows with too many such positions (heavy ties), or whose list would hold
// half the row or more (short rows), refine and emit over all keys instead:
// the emit pass gives each warp a contiguous segment of positions, counts per
// warp, scans the 32 warp counts once, and writes each warp's selections in
// order with ballots.  Two instantiations: two CTAs per SM (32 registers) for
// rows whose keys fit twice in shared memory, one CTA per SM otherwise.
//
// topk_kernel (any row length; used for rows longer than the shared-memory
// capacity, e.g. long decode caches): one CTA (1024 threads) per row.  Scores
// become order-preserving 32-bit keys (score_key).  Three histogram passes over
// 11 + 11 + 10 key bits find the exact key T of the k-th largest score and how many of the
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

constexpr int kTopkSmemKeys = 50 * 1024;   // keys held in shared memory (200 KB)
constexpr int kTopkBins = 2048;
constexpr int kTopkCand = 4096;            // candidate positions kept for the refining passes

__host__ __device__ constexpr size_t topk_smem_bytes(int max_len) {
    return static_cast<size_t>((max_len + 3) / 4 * 4) * 4 + kTopkBins * 4 + kTopkCand * 4 + 64 * 4 + 64;
}

// Prefetches `bytes` (a multiple of 16, 16-byte aligned source) of global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Persistent: CTA c takes rows c, c + gridDim.x, ...  One thread prefetches the CTA's next row
// into L2 while the current row is processed, so the HBM read of a row overlaps the work on the
// previous one.
//
// Per row:
//   pass 1   reads the row (the only HBM read of it), keeps its order-preserving keys in shared
//            memory and counts the top 11 key bits;
//   then     the bin B holding the k-th largest key is found.  Every key above the row's k-th
//            largest has top bits >= B, so when the keys with top bits >= B ("candidates") are
//            few, one ordered pass writes their positions, in position order, to a list, and the
//            two refining radix passes and the emit run over that list only.  Rows with more
//            candidates than the list holds (heavy ties), or with at least half their keys
//            listed (short rows), take the same passes over all keys.
//
// kMinBlocks = 2 caps registers at 32 so that two CTAs share an SM (rows short enough for two
// CTAs' shared memory); kMinBlocks = 1 leaves the compiler 64 registers for long rows.
template <int kMinBlocks>
__global__ void __launch_bounds__(kTopkThreads, kMinBlocks)
topk_smem_kernel(RowSpec rs, const float* __restrict__ scores, long long ld, int k, int rows,
                 int* __restrict__ idx_out) {
    extern __shared__ __align__(16) uint8_t tk_smem[];
    const int n_cap = (rs.max_len + 3) / 4 * 4;
    uint32_t* keys = reinterpret_cast<uint32_t*>(tk_smem);
    uint32_t* hist = keys + n_cap;
    uint32_t* cand = hist + kTopkBins;             // candidate positions, ascending
    uint32_t* s_cnt = cand + kTopkCand;            // [32] gt counts, [32] eq counts per warp
    uint32_t* s_misc = s_cnt + 64;                 // digit, keys above it, its count
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint4* keys4 = reinterpret_cast<uint4*>(keys);

    // Finds, from the histogram of `nb` bins, the bin holding the need-th largest key, the
    // number of keys above it and the bin's own count (thread t owns bins from the top).
    auto find_bin = [&](int nb, uint32_t need, uint32_t* digit, uint32_t* above_out, uint32_t* count) {
        const int per = nb / kTopkThreads;   // 2 or 1
        uint32_t cnt[2] = {0u, 0u};
        for (int e = 0; e < per; ++e) cnt[e] = hist[nb - 1 - tid * per - e];
        uint32_t tot;
        uint32_t above = block_excl_scan(cnt[0] + cnt[1], s_cnt, &tot);
        for (int e = 0; e < per; ++e) {
            if (above < need && need <= above + cnt[e]) {
                s_misc[0] = static_cast<uint32_t>(nb - 1 - tid * per - e);
                s_misc[1] = above;
                s_misc[2] = cnt[e];
            }
            above += cnt[e];
        }
        __syncthreads();
        *digit = s_misc[0];
        *above_out = s_misc[1];
        *count = s_misc[2];
        __syncthreads();
    };

    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        int* out = idx_out + static_cast<long long>(r) * k;
        const RowInfo ri = row_info(rs, r);
        const int n = ri.ok ? ri.n : 0;
        if (tid == 0 && r + static_cast<int>(gridDim.x) < rows) {
            const RowInfo rn = row_info(rs, r + gridDim.x);
            const int nn = rn.ok ? rn.n : 0;
            if (nn > k)
                prefetch_l2_bulk(scores + static_cast<long long>(r + gridDim.x) * ld,
                                 static_cast<uint32_t>((nn + 3) / 4) * 16u);
        }
        if (n <= k) {  // every candidate is kept (or the row is invalid: all -1)
            for (int i = tid; i < k; i += kTopkThreads) out[i] = (i < n) ? i : -1;
            continue;
        }
        const float4* row4 = reinterpret_cast<const float4*>(scores + static_cast<long long>(r) * ld);
        const int n4 = (n + 3) >> 2;

        // pass 1: keys to shared memory, histogram of the top 11 bits
        for (int i = tid; i < kTopkBins; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        for (int i4 = tid; i4 < n4; i4 += kTopkThreads) {
            const float4 v = __ldcs(row4 + i4);        // streamed: every score is read once from DRAM
            uint4 kk = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
            const int base = i4 * 4;
            if (base + 3 >= n) {   // the row's ragged tail: positions past n rank below everything
                if (base + 1 >= n) kk.y = 0u;
                if (base + 2 >= n) kk.z = 0u;
                if (base + 3 >= n) kk.w = 0u;
            }
            keys4[i4] = kk;
            atomicAdd(&hist[kk.x >> 21], 1u);
            if (base + 1 < n) atomicAdd(&hist[kk.y >> 21], 1u);
            if (base + 2 < n) atomicAdd(&hist[kk.z >> 21], 1u);
            if (base + 3 < n) atomicAdd(&hist[kk.w >> 21], 1u);
        }
        __syncthreads();
        uint32_t prefix, above, in_bin;
        find_bin(kTopkBins, static_cast<uint32_t>(k), &prefix, &above, &in_bin);
        uint32_t need = static_cast<uint32_t>(k) - above;
        const uint32_t ncand = above + in_bin;           // keys with top bits >= prefix
        // the list pays for its extra ordered pass only when it is well shorter than the row
        const bool listed = ncand <= static_cast<uint32_t>(kTopkCand) && 2 * ncand <= static_cast<uint32_t>(n);
        // warp w owns positions [w*seg, (w+1)*seg)
        const int seg = ((n4 + 31) / 32) * 4;
        const int p0 = wid * seg, p1 = min(n, p0 + seg);
        if (listed) {
            // the candidates' positions, in position order: warp w owns the 4-key groups
            // [w*seg4, (w+1)*seg4); a lane takes one group (16 bytes) per step
            const uint32_t B = prefix;
            const int seg4 = (n4 + 31) / 32;
            const int u0 = wid * seg4, u1 = min(n4, u0 + seg4);
            auto flags = [&](int u, uint32_t (&f)[4]) {
                const uint4 kk = (u < u1) ? keys4[u] : make_uint4(0u, 0u, 0u, 0u);
                const int p = 4 * u;
                f[0] = (u < u1 && (kk.x >> 21) >= B) ? 1u : 0u;
                f[1] = (u < u1 && p + 1 < n && (kk.y >> 21) >= B) ? 1u : 0u;
                f[2] = (u < u1 && p + 2 < n && (kk.z >> 21) >= B) ? 1u : 0u;
                f[3] = (u < u1 && p + 3 < n && (kk.w >> 21) >= B) ? 1u : 0u;
            };
            uint32_t c = 0;
            for (int u = u0 + lane; u < u1; u += 32) {
                uint32_t f[4];
                flags(u, f);
                c += f[0] + f[1] + f[2] + f[3];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (lane == 0) s_cnt[wid] = c;
            __syncthreads();
            uint32_t before = 0;
            for (int w = 0; w < wid; ++w) before += s_cnt[w];
            for (int base = u0; base < u1; base += 32) {
                const int u = base + lane;
                uint32_t f[4];
                flags(u, f);
                const uint32_t cnt = f[0] + f[1] + f[2] + f[3];
                uint32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t slot = before + incl - cnt;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (f[e]) cand[slot++] = static_cast<uint32_t>(4 * u + e);
                before += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncthreads();
        }
        // passes 2 and 3: the next 11 and 10 bits, over the keys that match the prefix found so far
#pragma unroll 1
        for (int pass = 1; pass < 3; ++pass) {
            const int shift = (pass == 1) ? 10 : 0;
            const int bits = (pass == 2) ? 10 : 11;
            const int nb = 1 << bits;
            const int hi_shift = shift + bits;
            const uint32_t mask = static_cast<uint32_t>(nb - 1);
            for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0u;
            __syncthreads();
            if (listed) {
                for (int j = tid; j < static_cast<int>(ncand); j += kTopkThreads) {
                    const uint32_t kk = keys[cand[j]];
                    if ((kk >> hi_shift) == prefix) atomicAdd(&hist[(kk >> shift) & mask], 1u);
                }
            } else {
                for (int i4 = tid; i4 < n4; i4 += kTopkThreads) {
                    const uint4 kk = keys4[i4];
                    const int base = i4 * 4;
                    if ((kk.x >> hi_shift) == prefix) atomicAdd(&hist[(kk.x >> shift) & mask], 1u);
                    if ((kk.y >> hi_shift) == prefix && base + 1 < n) atomicAdd(&hist[(kk.y >> shift) & mask], 1u);
                    if ((kk.z >> hi_shift) == prefix && base + 2 < n) atomicAdd(&hist[(kk.z >> shift) & mask], 1u);
                    if ((kk.w >> hi_shift) == prefix && base + 3 < n) atomicAdd(&hist[(kk.w >> shift) & mask], 1u);
                }
            }
            __syncthreads();
            uint32_t digit, ab, nbin;
            find_bin(nb, need, &digit, &ab, &nbin);
            (void)nbin;
            prefix = (prefix << bits) | digit;
            need -= ab;
        }
        const uint32_t T = prefix;   // key of the k-th largest score; `need` keys equal to T are kept

        if (listed) {
            // emit over the candidate list (position order): keys > T and the first `need` == T.
            // Warp w owns list entries [w*segc, (w+1)*segc): count, scan the warp counts, write.
            const int segc = (static_cast<int>(ncand) + 31) / 32;
            const int j0 = wid * segc, j1 = min(static_cast<int>(ncand), j0 + segc);
            uint32_t c_gt = 0, c_eq = 0;
            for (int j = j0 + lane; j < j1; j += 32) {
                const uint32_t kk = keys[cand[j]];
                c_gt += (kk > T) ? 1u : 0u;
                c_eq += (kk == T) ? 1u : 0u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                c_gt += __shfl_xor_sync(0xffffffffu, c_gt, o);
                c_eq += __shfl_xor_sync(0xffffffffu, c_eq, o);
            }
            if (lane == 0) { s_cnt[wid] = c_gt; s_cnt[32 + wid] = c_eq; }
            __syncthreads();
            uint32_t gt_before = 0, eq_before = 0;
            for (int w = 0; w < wid; ++w) { gt_before += s_cnt[w]; eq_before += s_cnt[32 + w]; }
            for (int base = j0; base < j1; base += 32) {
                const int j = base + lane;
                const uint32_t p = (j < j1) ? cand[j] : 0u;
                const uint32_t kk = (j < j1) ? keys[p] : 0u;
                const bool gt = (j < j1) && kk > T;
                const bool eq = (j < j1) && kk == T;
                const uint32_t mgt = __ballot_sync(0xffffffffu, gt), meq = __ballot_sync(0xffffffffu, eq);
                const uint32_t lt_mask = (1u << lane) - 1u;
                const uint32_t my_eq = eq_before + __popc(meq & lt_mask);       // equal keys before p
                if (gt || (eq && my_eq < need))
                    out[gt_before + __popc(mgt & lt_mask) + min(my_eq, need)] = static_cast<int>(p);
                gt_before += __popc(mgt);
                eq_before += __popc(meq);
            }
        } else {
            // emit over all keys: count per warp, scan the warp counts, write in order
            uint32_t c_gt = 0, c_eq = 0;
            for (int p = p0 + lane; p < p1; p += 32) {
                const uint32_t kk = keys[p];
                c_gt += (kk > T) ? 1u : 0u;
                c_eq += (kk == T) ? 1u : 0u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                c_gt += __shfl_xor_sync(0xffffffffu, c_gt, o);
                c_eq += __shfl_xor_sync(0xffffffffu, c_eq, o);
            }
            if (lane == 0) { s_cnt[wid] = c_gt; s_cnt[32 + wid] = c_eq; }
            __syncthreads();
            uint32_t gt_before = 0, eq_before = 0;
            for (int w = 0; w < wid; ++w) { gt_before += s_cnt[w]; eq_before += s_cnt[32 + w]; }
            for (int base = p0; base < p1; base += 32) {
                const int p = base + lane;
                const uint32_t kk = (p < p1) ? keys[p] : 0u;
                const bool gt = (p < p1) && kk > T;
                const bool eq = (p < p1) && kk == T;
                const uint32_t mgt = __ballot_sync(0xffffffffu, gt), meq = __ballot_sync(0xffffffffu, eq);
                const uint32_t lt_mask = (1u << lane) - 1u;
                const uint32_t my_eq = eq_before + __popc(meq & lt_mask);       // equal keys before p
                const bool take = gt || (eq && my_eq < need);
                if (take) {
                    const uint32_t slot = gt_before + __popc(mgt & lt_mask) + min(my_eq, need);
                    out[slot] = p;
                }
                gt_before += __popc(mgt);
                eq_before += __popc(meq);
            }
        }
        __syncthreads();   // shared memory is reused by the next row
    }
}

}  // namespace dsa
