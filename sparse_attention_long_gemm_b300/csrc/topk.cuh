// topk.cuh -- per-query top-k selection by radix select over fp32 scores.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", fine-grained token
// selection: keep the index_topk highest-scoring positions of each query
// (all of them when there are at most index_topk).  Equal scores go to the
// lower position.  Output: ascending positions, -1 padded.
//
// topk_rows_kernel (rows of at most kTkMaxLen positions): described below.
//
// topk_kernel (any row length; used only for rows longer than kTkMaxLen):
// one CTA (1024 threads) per row.  Scores
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

// ---------------------------------------------------------------------------
// topk_rows_kernel: rows of at most kTkMaxLen positions (every prefill row of
// the workloads here and decode caches up to 64 Ki positions).
//
// Persistent 256-thread CTAs, four or five per SM, one row at a time per CTA
// (rows r = blockIdx.x, + gridDim.x, ...), so that one CTA's barriers and
// scans overlap the others' streaming.  Per row of n > k scores:
//   1. threshold: the keys of 2048 positions spread evenly over the row (512
//      chunks of 4, copied into shared memory by cp.async while the CTA is
//      still busy with its previous row) go through one radix pass over their
//      top 11 key bits (quarter octaves of the score), which finds the bin of
//      the sample of rank rho from the top; inside the bin the key is linear in
//      the score, so K_lo is interpolated from the bin's count.  rho sits 5
//      standard deviations above the sample rank the row's k-th score is
//      expected to have, so the k-th score lies above K_lo with high
//      probability (and the filter checks it).  When rho would exceed the
//      sample (short rows), every score is a candidate instead.  The CTA's
//      next row is prefetched into L2 meanwhile.
//   2. filter: one streaming pass over the row (its only read from HBM) keeps
//      every score whose key is >= K_lo: a float compare against K_lo's value
//      selects exactly those keys for finite scores.  Warp w owns 128-score
//      groups w, w+8, ... and appends its survivors' keys and positions to its
//      own 512-entry part of the candidate list by ballot and popc: no atomics
//      and no dependent chains across lanes.
//   3. exact select: radix passes over the candidates on key offsets from the
//      smallest candidate key, with digits of up to 11 bits from the top of the
//      candidates' actual key range (so the first pass spreads them over many
//      bins), narrow the k-th largest key down to a bin; once the bin holds at
//      most kTkSmall keys, they are ranked directly by (key descending, position
//      ascending).  Heavy ties run the passes down to the exact key and keep the
//      lowest positions among the keys equal to it.
//   4. emit: the selected positions are marked in an n-bit bitmap, so one scan
//      of its words (a block prefix sum of their bit counts) writes them in
//      ascending order; a second bitmap holds the keys equal to the k-th when
//      only some of them are kept (the lowest positions).  The positions are
//      staged in the (by then unused) candidate list and leave in coalesced
//      16-byte stores.
// When the candidates are fewer than k (the sample's rank-rho key lay above
// the row's k-th score) or overflow a warp's part of the list (heavy ties, or
// high scores bunched in one warp's groups), the row runs the exact full-row
// path instead: three 11/11/10-bit radix passes over the row (re-read from
// L2), then bitmaps built with warp ballots.
// ---------------------------------------------------------------------------
constexpr int kTkThreads = 256;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkCap = 4096;                   // candidate list capacity
constexpr int kTkWarpCap = kTkCap / kTkWarps;  // a warp's part of the list
constexpr int kTkMaxLen = 65536;               // longest row (positions stored in 16 bits)
constexpr int kTkSmall = 32;                   // bin size resolved by direct ranking
constexpr int kTkSampleChunks = 512;           // 4-score chunks sampled per row
constexpr int kTkUnroll = 4;                   // 128-score groups loaded ahead per warp

// Shared memory of topk_rows_kernel; the bitmaps (two of `bw` words) are sized for the longest
// row of the launch and hold at least the 2048-bin histogram, which aliases them.
struct TkSmem {
    static constexpr int OFF_CAND = 0;                           // uint2 [kTkCap] (score bits, then key; position)
    static constexpr int OFF_SAMP = OFF_CAND + kTkCap * 8;       // float4 [kTkSampleChunks] prefetched samples
    static constexpr int OFF_SMALL = OFF_SAMP + kTkSampleChunks * 16;  // uint2 [kTkSmall] (position, key)
    static constexpr int OFF_WCNT = OFF_SMALL + kTkSmall * 8;    // u32 [kTkWarps] candidates per warp
    static constexpr int OFF_SCAN = OFF_WCNT + kTkWarps * 4;     // u32 [2 * kTkWarps]
    static constexpr int OFF_MISC = OFF_SCAN + 2 * kTkWarps * 4; // u32 [8]
    static constexpr int OFF_BITS = OFF_MISC + 8 * 4;            // u32 [2 * bw] bitmaps / histogram
    __host__ __device__ static constexpr int bitmap_words(int max_len) {
        return ((max_len + 31) / 32 + 3) / 4 * 4 < 1024 ? 1024 : ((max_len + 31) / 32 + 3) / 4 * 4;
    }
    __host__ __device__ static constexpr int bytes(int max_len) { return OFF_BITS + 2 * bitmap_words(max_len) * 4; }
};
static_assert(TkSmem::OFF_BITS % 16 == 0 && TkSmem::OFF_SAMP % 16 == 0, "vector access alignment");

// Exclusive prefix sum of one value per thread over the 256-thread block; *total = block sum.
__device__ __forceinline__ uint32_t tk_scan(uint32_t v, uint32_t* s_scan, uint32_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[wid] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) {
        const uint32_t t = s_scan[w];
        before += (w < wid) ? t : 0u;
        tot += t;
    }
    *total = tot;
    __syncthreads();   // s_scan may be reused by the caller's next scan
    return before + x - v;
}

// Same for two values at once.
__device__ __forceinline__ void tk_scan2(uint32_t a, uint32_t b, uint32_t* s_scan, uint32_t* ea, uint32_t* eb) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, x, o), v = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) { x += u; y += v; }
    }
    if (lane == 31) { s_scan[wid] = x; s_scan[kTkWarps + wid] = y; }
    __syncthreads();
    uint32_t ba = 0, bb = 0;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) {
        if (w < wid) { ba += s_scan[w]; bb += s_scan[kTkWarps + w]; }
    }
    *ea = ba + x - a;
    *eb = bb + y - b;
    __syncthreads();
}

// From a histogram of nb bins (a power of two, at most 2048), the bin holding the rank-th
// largest element (1-based; the highest bin index first), the number of elements in higher
// bins and the bin's own count: s_misc[0..2].  Every thread calls it.  A thread owns up to 8
// consecutive bins, read as two 16-byte words (conflict-free).
__device__ __forceinline__ void tk_find_bin(const uint32_t* hist, int nb, uint32_t rank, uint32_t* s_scan,
                                            uint32_t* s_misc) {
    const int tid = threadIdx.x;
    const int per = nb >= kTkThreads ? nb / kTkThreads : 1;
    const int lo = nb - (tid + 1) * per;       // this thread's lowest bin; it owns [lo, lo + per)
    uint32_t c[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (lo >= 0) {
        if (per == 8) {
            const uint4 a = reinterpret_cast<const uint4*>(hist + lo)[0], b = reinterpret_cast<const uint4*>(hist + lo)[1];
            c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w; c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < per) c[e] = hist[lo + e];
        }
    }
    uint32_t sum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) sum += c[e];
    uint32_t tot;
    uint32_t above = tk_scan(sum, s_scan, &tot);   // elements in higher bins than this thread's
    if (lo >= 0 && above < rank && rank <= above + sum) {
#pragma unroll
        for (int e = 7; e >= 0; --e) {
            if (e < per) {
                if (rank <= above + c[e]) {
                    s_misc[0] = static_cast<uint32_t>(lo + e);
                    s_misc[1] = above;
                    s_misc[2] = c[e];
                    break;
                }
                above += c[e];
            }
        }
    }
    __syncthreads();
}

// Shared-memory reductions that do nothing when `p` is false (predicated, so that loops over
// candidates stay free of divergent branches).
__device__ __forceinline__ void red_add_shared_if(bool p, const uint32_t* addr, uint32_t v) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t@q red.shared.add.u32 [%1], %2;\n\t}"
                 ::"r"(static_cast<uint32_t>(p)), "r"(smem_u32(addr)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_shared_if(bool p, const uint32_t* addr, uint32_t v) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %0, 0;\n\t@q red.shared.or.b32 [%1], %2;\n\t}"
                 ::"r"(static_cast<uint32_t>(p)), "r"(smem_u32(addr)), "r"(v) : "memory");
}

// Inverse of score_key for keys of finite scores: the float whose key is `key`.
__device__ __forceinline__ float tk_key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Number of positions of a row of n >= 1 scores that the sample covers, and the row chunk of
// sample chunk j (chunks spread evenly over the row's n4 = ceil(n / 4) chunks).
__device__ __forceinline__ int tk_sample_chunks(int n) { return min(kTkSampleChunks, (n + 3) >> 2); }
__device__ __forceinline__ int tk_sample_chunk(int j, int ms4, int n4) {
    return static_cast<int>((static_cast<uint32_t>(j) * static_cast<uint32_t>(n4)) / static_cast<uint32_t>(ms4));
}

// Issues the cp.async copies of row r's sample chunks into the sample buffer (no wait).
__device__ __forceinline__ void tk_prefetch_samples(const RowSpec& rs, const float* scores, long long ld, int k,
                                                    int r, uint32_t s_samp) {
    const RowInfo ri = row_info(rs, r);
    const int n = ri.ok ? ri.n : 0;
    if (n > k) {
        const int n4 = (n + 3) >> 2, ms4 = tk_sample_chunks(n);
        const float* row = scores + static_cast<long long>(r) * ld;
        for (int j = threadIdx.x; j < ms4; j += kTkThreads)
            cp_async_16(s_samp + 16u * j, row + 4 * tk_sample_chunk(j, ms4, n4));
    }
    cp_async_commit();
}

// Prefetches row r's scores (if it needs selecting) from HBM into L2 with one bulk request.
__device__ __forceinline__ void tk_prefetch_row_l2(const RowSpec& rs, const float* scores, long long ld, int k, int r) {
    const RowInfo ri = row_info(rs, r);
    if (ri.ok && ri.n > k)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(scores + static_cast<long long>(r) * ld), "r"(static_cast<uint32_t>((ri.n + 3) / 4) * 16u)
                     : "memory");
}

#ifndef DSA_TOPK_MIN_BLOCKS
#define DSA_TOPK_MIN_BLOCKS 4
#endif
__global__ void __launch_bounds__(kTkThreads, DSA_TOPK_MIN_BLOCKS)
topk_rows_kernel(RowSpec rs, const float* __restrict__ scores, long long ld, int k, int rows,
                 int* __restrict__ idx_out) {
    extern __shared__ __align__(16) uint8_t tk_smem[];
    uint2* cand = reinterpret_cast<uint2*>(tk_smem + TkSmem::OFF_CAND);
    const float4* samp = reinterpret_cast<const float4*>(tk_smem + TkSmem::OFF_SAMP);
    uint2* small = reinterpret_cast<uint2*>(tk_smem + TkSmem::OFF_SMALL);
    uint32_t* wcnt = reinterpret_cast<uint32_t*>(tk_smem + TkSmem::OFF_WCNT);
    uint32_t* s_scan = reinterpret_cast<uint32_t*>(tk_smem + TkSmem::OFF_SCAN);
    uint32_t* s_misc = reinterpret_cast<uint32_t*>(tk_smem + TkSmem::OFF_MISC);
    const int bw = TkSmem::bitmap_words(rs.max_len);
    uint32_t* gtb = reinterpret_cast<uint32_t*>(tk_smem + TkSmem::OFF_BITS);
    uint32_t* eqb = gtb + bw;
    uint32_t* hist = gtb;                          // 2048 bins over both bitmaps (bw >= 1024)
    uint32_t* skey = reinterpret_cast<uint32_t*>(cand);   // sample keys (before the filter)
    int* stage = reinterpret_cast<int*>(cand);            // the emitted positions (after the select)
    const bool staged = k <= 2 * kTkCap;
    const uint32_t s_samp = smem_u32(tk_smem + TkSmem::OFF_SAMP);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    const bool list_ok = 2 * k <= kTkCap;          // the candidate list can hold k plus a margin

    if (blockIdx.x < rows) {
        if (tid == 0) tk_prefetch_row_l2(rs, scores, ld, k, blockIdx.x);
        if (list_ok) tk_prefetch_samples(rs, scores, ld, k, blockIdx.x, s_samp);
    }
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        int* out = idx_out + static_cast<long long>(r) * k;
        const RowInfo ri = row_info(rs, r);
        const int n = ri.ok ? ri.n : 0;
        // the next row streams from HBM into L2 while this one is worked on
        if (tid == 0 && r + static_cast<int>(gridDim.x) < rows) tk_prefetch_row_l2(rs, scores, ld, k, r + gridDim.x);
        if (list_ok) cp_async_wait<0>();           // this row's samples (if any) have landed
        __syncthreads();
        if (n <= k) {   // every candidate is kept (or the row is invalid: all -1)
            for (int i = tid; i < k; i += kTkThreads) out[i] = (i < n) ? i : -1;
            if (list_ok && r + static_cast<int>(gridDim.x) < rows)
                tk_prefetch_samples(rs, scores, ld, k, r + gridDim.x, s_samp);
            continue;
        }
        const float* row = scores + static_cast<long long>(r) * ld;
        const float4* row4 = reinterpret_cast<const float4*>(row);
        const int n4 = (n + 3) >> 2;
        const int nw = (n + 31) >> 5;
        bool full_row = !list_ok;
        bool take_all = false;
        uint32_t klo = 0, smax = 0;    // filter threshold key; largest sampled key

        // ---------------- 1. threshold from the sample ----------------
        if (!full_row) {
            const int ms4 = tk_sample_chunks(n);
            const int m = 4 * ms4;
            const float mp = static_cast<float>(m) * static_cast<float>(k) / static_cast<float>(n);
            const uint32_t rho = static_cast<uint32_t>(ceilf(mp + 5.f * sqrtf(mp) + 2.f));
            if (rho >= static_cast<uint32_t>(m)) {
                take_all = n <= kTkCap;
                full_row = !take_all;
            } else {
                uint32_t smx = 0;
                for (int j = tid; j < ms4; j += kTkThreads) {
                    const float4 v = samp[j];
                    const int p = 4 * tk_sample_chunk(j, ms4, n4);
                    uint4 kk = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
                    if (p + 1 >= n) kk.y = 0u;   // positions past the row rank lowest
                    if (p + 2 >= n) kk.z = 0u;
                    if (p + 3 >= n) kk.w = 0u;
                    reinterpret_cast<uint4*>(skey)[j] = kk;
                    smx = max(smx, max(max(kk.x, kk.y), max(kk.z, kk.w)));
                }
                smx = __reduce_max_sync(0xffffffffu, smx);
                // one radix pass over the top 11 key bits (quarter octaves of the score), then the
                // rank-rho key is interpolated inside its bin, where the key is linear in the score
                for (int i = tid; i < 512; i += kTkThreads) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
                if (tid == 0) s_misc[3] = 0u;
                __syncthreads();
                if (lane == 0) atomicMax(&s_misc[3], smx);
                for (int j = tid; j < m; j += kTkThreads) {
                    const uint32_t kk = skey[j];
                    atomicAdd(&hist[kk >> 21], 1u);
                }
                __syncthreads();
                tk_find_bin(hist, 2048, rho, s_scan, s_misc);
                const uint32_t bin = s_misc[0], want = rho - s_misc[1], inbin = s_misc[2];
                smax = s_misc[3];
                __syncthreads();
                // the bin holds `inbin` samples spread over 2^21 keys; `want` of them from its top
                const uint32_t drop = static_cast<uint32_t>((static_cast<unsigned long long>(want) << 21) / inbin);
                const unsigned long long top = static_cast<unsigned long long>(bin + 1u) << 21;   // <= 2^32
                klo = static_cast<uint32_t>(min(top - min(drop, 1u << 21), 0xffffffffull)) & ~1023u;
                if (klo == 0u) full_row = true;   // no usable threshold (a sample dominated by NaN)
            }
        }

        // ---------------- 2. filter into the candidate list ----------------
        uint32_t c_tot = 0, kmin_all = 0, kmax_all = 0;
        if (!full_row) {
            if (tid == 0) { s_misc[4] = 0u; s_misc[5] = 0xffffffffu; s_misc[7] = 0u; }
            uint32_t cnt = 0, kmin = 0xffffffffu, kmax = 0u;
            uint2* wc = cand + wid * kTkWarpCap;
            const int ngroups = (n + 127) >> 7;       // 128 scores per group: 32 lanes x float4
            if (take_all) {
                // every score is a candidate (NaN too: its key ranks lowest); exact key range
#pragma unroll 1
                for (int g = wid; g < ngroups; g += kTkWarps) {
                    const int c = g * 32 + lane;
                    const float4 v = (c < n4) ? __ldcs(row4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const int p = 4 * c;
                    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool pr = p + q < n;
                        const uint32_t m = __ballot_sync(0xffffffffu, pr);
                        const uint32_t slot = cnt + __popc(m & lt);
                        const uint32_t kk = score_key(e[q]);
                        if (pr && slot < static_cast<uint32_t>(kTkWarpCap))
                            wc[slot] = make_uint2(__float_as_uint(e[q]), static_cast<uint32_t>(p + q));
                        kmin = pr ? min(kmin, kk) : kmin;
                        kmax = pr ? max(kmax, kk) : kmax;
                        cnt += __popc(m);
                    }
                }
            } else {
                // scores >= tau, the float whose key is K_lo; positions past the row read as -inf
                const float tau = tk_key_float(klo);
#pragma unroll 1
                for (int g0 = wid; g0 < ngroups; g0 += kTkWarps * kTkUnroll) {
                    float4 v[kTkUnroll];
#pragma unroll
                    for (int u = 0; u < kTkUnroll; ++u) {
                        const int c = (g0 + u * kTkWarps) * 32 + lane;
                        v[u] = (c < n4) ? __ldcs(row4 + c) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                        const int lim = n - 4 * c;    // valid scores in this chunk, when fewer than 4
                        if (lim < 4) {
                            if (lim < 2) v[u].y = -INFINITY;
                            if (lim < 3) v[u].z = -INFINITY;
                            v[u].w = -INFINITY;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kTkUnroll; ++u) {
                        const uint32_t p = static_cast<uint32_t>(4 * ((g0 + u * kTkWarps) * 32 + lane));
                        const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const bool pr = e[q] >= tau;
                            const uint32_t m = __ballot_sync(0xffffffffu, pr);
                            const uint32_t slot = cnt + __popc(m & lt);
                            if (pr && slot < static_cast<uint32_t>(kTkWarpCap))
                                wc[slot] = make_uint2(__float_as_uint(e[q]), p + q);
                            cnt += __popc(m);
                        }
                    }
                }
            }
            kmin = __reduce_min_sync(0xffffffffu, kmin);
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            __syncthreads();   // the misc words are initialised
            if (lane == 0) {
                wcnt[wid] = min(cnt, static_cast<uint32_t>(kTkWarpCap));
                if (take_all) {
                    atomicMax(&s_misc[4], kmax);
                    atomicMin(&s_misc[5], kmin);
                }
                atomicAdd(&s_misc[7], cnt);
                if (cnt > static_cast<uint32_t>(kTkWarpCap)) atomicOr(&s_misc[7], 0x80000000u);   // overflow
            }
            __syncthreads();
            c_tot = s_misc[7];
            kmax_all = s_misc[4];
            kmin_all = s_misc[5];
            if ((c_tot & 0x80000000u) || c_tot < static_cast<uint32_t>(k)) full_row = true;
        }
        // the next row's samples go into their buffer while this row is finished (every thread
        // is past its reads of the buffer: rows that skip the filter reach here without a barrier)
        if (list_ok && r + static_cast<int>(gridDim.x) < rows) {
            __syncthreads();
            tk_prefetch_samples(rs, scores, ld, k, r + gridDim.x, s_samp);
        }

        uint32_t need = 0;   // keys equal to the k-th to keep (lowest positions), when they are tied
        if (!full_row) {
            // ---------------- 3. exact select over the candidates ----------------
            // Digits are taken from key offsets o = key - base.  take_all: base and range are the
            // exact key range.  Sampled: base = K_lo (every candidate's key is >= K_lo) and the
            // range is twice the offset of the largest sampled key; the few candidates beyond it
            // fall into the first pass's top bin (clamped), which is fine unless the k-th key is
            // there, and then the row takes the exact full-row path.
            uint32_t base, range;
            if (take_all) {
                base = kmin_all;
                range = kmax_all - base;
            } else {
                base = klo;
                range = static_cast<uint32_t>(min(2ull * (smax - klo) + 1ull, 0xffffffffull));
            }
            int shift = range ? 32 - __clz(range) : 0;   // the prefix so far is offset >> shift
            uint32_t prefix = 0, rank = static_cast<uint32_t>(k), cnt = c_tot;
            if (cnt <= static_cast<uint32_t>(kTkSmall)) shift = 32;   // one bin: rank them all directly
            // this thread visits slots j = tid + 256 i of the list: part i / 2, entry 256 (i & 1) + tid
            constexpr int kSlots = kTkCap / kTkThreads;
            static_assert(kTkWarpCap == 2 * kTkThreads, "two visits per warp part");
            uint32_t wcr[kTkWarps];
#pragma unroll
            for (int w = 0; w < kTkWarps; ++w) wcr[w] = wcnt[w];
            auto valid = [&](int i) { return static_cast<uint32_t>(kTkThreads * (i & 1) + tid) < wcr[i >> 1]; };
            // the candidates' keys replace their score bits (each thread converts the slots it visits)
#pragma unroll
            for (int i = 0; i < kSlots; ++i) {
                uint32_t* x = &cand[tid + kTkThreads * i].x;
                *x = score_key(__uint_as_float(*x));
            }
            bool first = true;
#pragma unroll 1
            while (shift > 0 && cnt > static_cast<uint32_t>(kTkSmall)) {
                const int ns = max(shift - 11, 0), width = shift - ns, nb = 1 << width;
                for (int i = tid; i < (nb >> 2); i += kTkThreads) reinterpret_cast<uint4*>(hist)[i] = make_uint4(0u, 0u, 0u, 0u);
                if (nb < 4 && tid < nb) hist[tid] = 0u;
                __syncthreads();
#pragma unroll
                for (int i = 0; i < kSlots; ++i) {
                    const uint32_t o = cand[tid + kTkThreads * i].x - base;
                    const bool el = valid(i) && (first || (o >> shift) == prefix);
                    const uint32_t dg = first ? min(o >> ns, static_cast<uint32_t>(nb - 1)) : ((o >> ns) & (nb - 1));
                    red_add_shared_if(el, &hist[dg], 1u);
                }
                __syncthreads();
                tk_find_bin(hist, nb, rank, s_scan, s_misc);
                const uint32_t dig = s_misc[0];
                if (first && !take_all && dig == static_cast<uint32_t>(nb - 1)) {   // the k-th is past the range
                    full_row = true;
                    __syncthreads();
                    break;
                }
                prefix = (prefix << width) | dig;
                rank -= s_misc[1];
                cnt = s_misc[2];
                shift = ns;
                first = false;
                __syncthreads();
            }
            if (!full_row) {
                // mark: candidates in higher bins are selected; the bin's own are ranked directly when
                // few, else (all equal: shift == 0) kept lowest position first
                const bool few = cnt <= static_cast<uint32_t>(kTkSmall);
                for (int i = tid; i < bw / 2; i += kTkThreads) reinterpret_cast<uint4*>(gtb)[i] = make_uint4(0u, 0u, 0u, 0u);
                if (tid == 0) s_misc[6] = 0u;
                __syncthreads();
#pragma unroll
                for (int i = 0; i < kSlots; ++i) {
                    const uint2 cj = cand[tid + kTkThreads * i];
                    const bool v = valid(i);
                    const uint32_t kk = cj.x;
                    const uint32_t o = kk - base;
                    const uint32_t d = shift >= 32 ? 0u : (o >> shift);
                    const uint32_t p = cj.y;
                    red_or_shared_if(v && d > prefix, &gtb[p >> 5], 1u << (p & 31));
                    red_or_shared_if(v && !few && d == prefix, &eqb[p >> 5], 1u << (p & 31));
                    if (v && few && d == prefix) {   // at most kTkSmall lanes of the CTA take this
                        const uint32_t si = atomicAdd(&s_misc[6], 1u);
                        if (si < static_cast<uint32_t>(kTkSmall)) small[si] = make_uint2(p, kk);
                    }
                }
                __syncthreads();
                if (few) {
                    if (wid == 0 && lane < static_cast<int>(cnt)) {
                        const uint2 me = small[lane];
                        uint32_t before = 0;
                        for (int j = 0; j < static_cast<int>(cnt); ++j) {
                            const uint2 o = small[j];
                            before += (o.y > me.y || (o.y == me.y && o.x < me.x)) ? 1u : 0u;
                        }
                        if (before < rank) atomicOr(&gtb[me.x >> 5], 1u << (me.x & 31));
                    }
                    __syncthreads();
                } else {
                    need = rank;
                }
            }
        }
        if (full_row) {
            // ---------------- exact full-row path ----------------
            uint32_t prefix = 0, rank = static_cast<uint32_t>(k);
#pragma unroll 1
            for (int pass = 0; pass < 3; ++pass) {
                const int shift = (pass == 0) ? 21 : (pass == 1 ? 10 : 0);
                const int bits = (pass == 2) ? 10 : 11;
                const int nb = 1 << bits;
                const int hi = shift + bits;
                for (int i = tid; i < nb; i += kTkThreads) hist[i] = 0u;
                __syncthreads();
                for (int c0 = 0; c0 < n4; c0 += kTkThreads) {   // warp-uniform trip count
                    const int c = c0 + tid;
                    const float4 v = (c < n4) ? __ldg(row4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const int p = 4 * c;
                    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // lanes with the same bin add once together (rows reaching this path are often
                        // full of equal keys, which would serialise one atomic per lane)
                        const uint32_t kk = score_key(e[q]);
                        const bool in = p + q < n && (pass == 0 || (kk >> hi) == prefix);
                        const uint32_t bin = in ? ((kk >> shift) & (nb - 1)) : 0xffffffffu;
                        const uint32_t grp = __match_any_sync(0xffffffffu, bin);
                        if (in && lane == __ffs(grp) - 1) atomicAdd(&hist[bin], __popc(grp));
                    }
                }
                __syncthreads();
                tk_find_bin(hist, nb, rank, s_scan, s_misc);
                prefix = (prefix << bits) | s_misc[0];
                rank -= s_misc[1];
                __syncthreads();
            }
            const uint32_t T = prefix;
            need = rank;
            // bitmaps by ballot: word w holds positions 32w .. 32w+31 (also the words past nw up to
            // a multiple of 4, which the emit's 16-byte loads read: zero there)
            for (int w = wid; w < ((nw + 3) & ~3); w += kTkWarps) {
                const int p = 32 * w + lane;
                const uint32_t kk = (p < n) ? score_key(__ldg(row + p)) : 0u;
                const uint32_t g = __ballot_sync(0xffffffffu, p < n && kk > T);
                const uint32_t q = __ballot_sync(0xffffffffu, p < n && kk == T);
                if (lane == 0) { gtb[w] = g; eqb[w] = q; }
            }
            __syncthreads();
        }

        // ---------------- 4. emit in position order ----------------
        {
            // thread t owns words [t W, t W + W): four at a time as 16-byte loads when W allows
            const int W = (nw + kTkThreads - 1) / kTkThreads;
            const int w0 = min(nw, tid * W), w1 = min(nw, w0 + W);
            uint32_t gs = 0, es = 0;
            if ((W & 3) == 0) {
                for (int w = w0; w < w1; w += 4) {   // the bitmaps are zero past nw up to a multiple of 4
                    const uint4 g = *reinterpret_cast<const uint4*>(gtb + w), q = *reinterpret_cast<const uint4*>(eqb + w);
                    gs += __popc(g.x) + __popc(g.y) + __popc(g.z) + __popc(g.w);
                    es += __popc(q.x) + __popc(q.y) + __popc(q.z) + __popc(q.w);
                }
            } else {
                for (int w = w0; w < w1; ++w) { gs += __popc(gtb[w]); es += __popc(eqb[w]); }
            }
            uint32_t g_before, e_before;
            tk_scan2(gs, es, s_scan, &g_before, &e_before);
            uint32_t slot = g_before + min(e_before, need);
            uint32_t eqc = e_before;
            for (int w = w0; w < w1; ++w) {
                uint32_t sel = gtb[w];
                uint32_t e = eqb[w];
                while (e) {   // equal keys: the lowest positions until `need` are kept
                    const uint32_t b = e & (0u - e);
                    if (eqc < need) sel |= b;
                    ++eqc;
                    e ^= b;
                }
                while (sel) {
                    const int b = __ffs(sel) - 1;
                    sel &= sel - 1;
                    if (slot < static_cast<uint32_t>(k)) {   // exactly k are marked; this only bounds writes
                        if (staged) stage[slot] = 32 * w + b;
                        else out[slot] = 32 * w + b;
                    }
                    ++slot;
                }
            }
            if (staged) {   // the row's k positions leave shared memory in coalesced stores
                __syncthreads();
                if ((k & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) {
                    for (int i = tid; i < (k >> 2); i += kTkThreads)
                        reinterpret_cast<int4*>(out)[i] = reinterpret_cast<const int4*>(stage)[i];
                } else {
                    for (int i = tid; i < k; i += kTkThreads) out[i] = stage[i];
                }
            }
        }
    }
    if (list_ok) cp_async_wait<0>();   // no copy is left in flight when the CTA exits
}

}  // namespace dsa
