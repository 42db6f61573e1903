// attn_bwd.cuh -- backward of the sparse MLA attention, the selection held fixed.
//
// DeepSeek-V3.2 page, overview: DSA is a trainable sparse attention.  The
// selection (top-k of the index scores) is piecewise constant, so the gradient
// reaches q and kv through the attention over the selected set only, which is
// plain softmax attention (absorbed MLA: one shared d_qk-wide key row per
// position, value = its first d_v columns).  For output gradients dO (and dlse):
//
//   D[h]     = dO[h,:] . O[h,:]
//   dz[h,i]  = p[h,i] * (dO[h,:] . kv[s_i,:d_v] - D[h] + dlse[h]),  p = exp(z - lse)
//   dq[h,:]  = scale * sum_i dz[h,i] kv[s_i,:]
//   dkv[s_i] += scale * sum_h dz[h,i] q[h,:]  (+ sum_h p[h,i] dO[h,:] on the value columns)
//
// One CTA per (query row, group of 32 heads), on the CUDA cores in fp32.  The
// query and output-gradient rows of the group stay in shared memory; the
// selected kv rows stream through a double-buffered tile of 32 rows (cp.async
// gathers of block b+1 overlap the arithmetic of block b).  Per block:
//   A  logits and dP = dO . v  (32 heads x 32 keys; half the threads each)
//   B  p, dz                    (exp of the recomputed logit against the forward's lse)
//   C  dq += dz . kv            (kept in registers for the whole row)
//   D  dkv rows of the block    (fp32 atomic adds, two columns at a time)
#pragma once

#include "rows.cuh"

namespace dsa {

constexpr int kAbThreads = 256;
constexpr int kAbHeads = 32;      // heads per CTA
constexpr int kAbKeys = 32;       // selected positions per block
constexpr int kAbMaxPairs = 5;    // column pairs per thread in C and D: d_qk <= 2 * 64 * 5
constexpr int kAbMaxDqk = 2 * 64 * kAbMaxPairs;
constexpr int kAbSP = kAbKeys + 4;   // fp32 row stride of the [head][key] tiles (words = 4 mod 32)
constexpr int kAbST = kAbHeads + 4;  // fp32 row stride of the [key][head] tile

// Row stride (elements) of a shared tile of d columns of T: a whole number of 16-byte
// chunks whose word count is 4 mod 32, so that eight rows read at one column fall in
// eight distinct groups of banks.
template <typename T>
__host__ __device__ constexpr int ab_stride(int d) {
    return ((d * static_cast<int>(sizeof(T)) / 4 + 31) / 32 * 32 + 4) * 4 / static_cast<int>(sizeof(T));
}

template <typename T>
struct AbSmem {
    int sq, so;            // row strides (elements) of the q / kv tiles and of the dO tile
    size_t q, dout, kv, s, dp, p, dz, dzt, vec, idx, bytes;
    __host__ __device__ AbSmem(int d_qk, int d_v) {
        sq = ab_stride<T>(d_qk);
        so = ab_stride<T>(d_v);
        q = 0;
        dout = q + sizeof(T) * kAbHeads * sq;
        kv = dout + sizeof(T) * kAbHeads * so;
        s = kv + sizeof(T) * 2 * kAbKeys * sq;
        dp = s + sizeof(float) * kAbHeads * kAbSP;
        p = dp + sizeof(float) * kAbHeads * kAbSP;
        dz = p + sizeof(float) * kAbHeads * kAbSP;
        dzt = dz + sizeof(float) * kAbHeads * kAbSP;
        vec = dzt + sizeof(float) * kAbKeys * kAbST;   // D, lse, dlse: 3 x kAbHeads floats
        idx = vec + sizeof(float) * 3 * kAbHeads;      // 2 x kAbKeys positions
        bytes = idx + sizeof(int) * 2 * kAbKeys;
    }
};

__device__ __forceinline__ float2 ld_f2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld_f2(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Copies rows [0, nrows) of `src` (row stride `gstride` elements, `d` columns) into the
// shared tile at `dst` (row stride `sstride`); rows >= `valid` are zero-filled.
template <typename T>
__device__ __forceinline__ void ab_load_rows(T* dst, int sstride, const T* src, long long gstride, int d, int nrows,
                                             int valid, int tid) {
    const int cpr = d * static_cast<int>(sizeof(T)) / 16;   // 16-byte chunks per row
    constexpr int kPer = 16 / sizeof(T);
    for (int c = tid; c < nrows * cpr; c += kAbThreads) {
        const int row = c / cpr, part = c - row * cpr;
        T* d16 = dst + row * sstride + part * kPer;
        if (row < valid)
            cp_async_16(smem_u32(d16), src + row * gstride + part * kPer);
        else
            *reinterpret_cast<uint4*>(d16) = make_uint4(0u, 0u, 0u, 0u);
    }
}

template <typename T>
__global__ void __launch_bounds__(kAbThreads, 1)
attn_bwd_kernel(RowSpec rs, const T* __restrict__ q, const T* __restrict__ kv, const int* __restrict__ idx, int k,
                int H, int d_qk, int d_v, float scale, const T* __restrict__ out, const float* __restrict__ lse,
                const T* __restrict__ dout, const float* __restrict__ dlse, float* __restrict__ dq,
                float* __restrict__ dkv, int total_q) {
    extern __shared__ __align__(16) unsigned char smem[];
    const AbSmem<T> L(d_qk, d_v);
    T* sq = reinterpret_cast<T*>(smem + L.q);
    T* sdo = reinterpret_cast<T*>(smem + L.dout);
    T* skv = reinterpret_cast<T*>(smem + L.kv);
    float* sS = reinterpret_cast<float*>(smem + L.s);
    float* sdP = reinterpret_cast<float*>(smem + L.dp);
    float* sP = reinterpret_cast<float*>(smem + L.p);
    float* sdZ = reinterpret_cast<float*>(smem + L.dz);
    float* sdZt = reinterpret_cast<float*>(smem + L.dzt);
    float* sD = reinterpret_cast<float*>(smem + L.vec);
    float* slse = sD + kAbHeads;
    float* sdl = slse + kAbHeads;
    int* sidx = reinterpret_cast<int*>(smem + L.idx);
    const int SQ = L.sq, SO = L.so;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int r = total_q - 1 - static_cast<int>(blockIdx.x);   // longest rows of a sequence first
    const int h0 = blockIdx.y * kAbHeads;
    const int hn = min(kAbHeads, H - h0);                        // heads of this CTA
    const int pairs = d_qk >> 1, vpairs = d_v >> 1;
    const RowInfo ri = row_info(rs, r);
    if (!ri.ok) {   // lengths out of range (already raised): no gradient from this row
        for (int e = tid; e < hn * d_qk; e += kAbThreads) dq[(static_cast<long long>(r) * H + h0) * d_qk + e] = 0.f;
        return;
    }
    const int n = ri.n;
    const long long qrow = static_cast<long long>(r) * H + h0;   // first (row, head) of the CTA

    // Gathers the kv rows of selection block `b` into buffer `buf`; invalid or empty
    // entries become zero rows with position -1.
    const int cpr = d_qk * static_cast<int>(sizeof(T)) / 16;
    constexpr int kPer = 16 / sizeof(T);
    auto load_block = [&](int b, int buf) {
        T* dst = skv + buf * kAbKeys * SQ;
        for (int c = tid; c < kAbKeys * cpr; c += kAbThreads) {
            const int i = c / cpr, part = c - i * cpr;
            const int e = b * kAbKeys + i;
            const int s = e < k ? __ldg(idx + static_cast<long long>(r) * k + e) : -1;
            const bool valid = s >= 0 && s < n;
            if (part == 0) {
                if (!valid && s != -1) raise_error(DSA_ERR_DEVICE_DATA);
                sidx[buf * kAbKeys + i] = valid ? s : -1;
            }
            T* d16 = dst + i * SQ + part * kPer;
            if (valid)
                cp_async_16(smem_u32(d16), kv + (ri.key_base + s) * d_qk + part * kPer);
            else
                *reinterpret_cast<uint4*>(d16) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    ab_load_rows(sq, SQ, q + qrow * d_qk, d_qk, d_qk, kAbHeads, hn, tid);
    ab_load_rows(sdo, SO, dout + qrow * d_v, d_v, d_v, kAbHeads, hn, tid);
    load_block(0, 0);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // D = dO . O per head (a warp per head); lse of the forward (a non-finite lse, or a
    // head beyond H, gives p = 0); dlse (zero when absent)
    for (int h = wid; h < kAbHeads; h += kAbThreads / 32) {
        float acc = 0.f;
        if (h < hn) {
            const T* orow = out + (qrow + h) * d_v;
            for (int c = lane; c < d_v; c += 32) acc = fmaf(to_f32(sdo[h * SO + c]), to_f32(orow[c]), acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            sD[h] = acc;
            const float l = h < hn ? __ldg(lse + qrow + h) : INFINITY;
            slse[h] = isfinite(l) ? l : INFINITY;
            sdl[h] = (h < hn && dlse != nullptr) ? __ldg(dlse + qrow + h) : 0.f;
        }
    }

    // C's accumulators: heads 8*hq .. 8*hq+7, column pairs cl + 64*j
    const int hq = tid >> 6, cl = tid & 63;
    float2 acc_dq[8][kAbMaxPairs];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int j = 0; j < kAbMaxPairs; ++j) acc_dq[a][j] = make_float2(0.f, 0.f);

    const int nb = (k + kAbKeys - 1) / kAbKeys;
    for (int b = 0; b < nb; ++b) {
        const int buf = b & 1;
        if (b + 1 < nb) load_block(b + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        // block b's rows and positions are in place; a block with no valid entry is skipped
        if (!__syncthreads_or(tid < kAbKeys && sidx[buf * kAbKeys + tid] >= 0)) continue;
        const T* kvb = skv + buf * kAbKeys * SQ;
        const int* ib = sidx + buf * kAbKeys;

        // A: raw logits q.kv (threads 0..127) and dP = dO.v (threads 128..255);
        //    heads hb + 8*a, keys kb and kb + 16
        {
            const int u = tid & 127, hb = u & 7, kb = u >> 3;
            const bool is_s = tid < 128;
            const T* arow = is_s ? sq : sdo;
            const int as = is_s ? SQ : SO;
            const int dd = is_s ? d_qk : d_v;
            float acc[4][2];
#pragma unroll
            for (int a = 0; a < 4; ++a) acc[a][0] = acc[a][1] = 0.f;
            for (int c = 0; c < dd; c += 2) {
                const float2 k0 = ld_f2(kvb + kb * SQ + c);
                const float2 k1 = ld_f2(kvb + (kb + 16) * SQ + c);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const float2 x = ld_f2(arow + (hb + 8 * a) * as + c);
                    acc[a][0] = fmaf(x.x, k0.x, fmaf(x.y, k0.y, acc[a][0]));
                    acc[a][1] = fmaf(x.x, k1.x, fmaf(x.y, k1.y, acc[a][1]));
                }
            }
            float* dst = is_s ? sS : sdP;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                dst[(hb + 8 * a) * kAbSP + kb] = acc[a][0];
                dst[(hb + 8 * a) * kAbSP + kb + 16] = acc[a][1];
            }
        }
        __syncthreads();

        // B: p = exp(scale * logit - lse), dz = scale * p * (dP - D + dlse); both layouts of dz
        for (int e = tid; e < kAbHeads * kAbKeys; e += kAbThreads) {
            const int h = e / kAbKeys, i = e - h * kAbKeys;
            float p = 0.f, dz = 0.f;
            if (ib[i] >= 0) {
                p = expf(fmaf(sS[h * kAbSP + i], scale, -slse[h]));
                dz = scale * p * (sdP[h * kAbSP + i] - sD[h] + sdl[h]);
            }
            sP[h * kAbSP + i] = p;
            sdZ[h * kAbSP + i] = dz;
            sdZt[i * kAbST + h] = dz;
        }
        __syncthreads();

        // C: dq[h, :] += sum_i dz[h, i] kv[i, :]
        for (int i = 0; i < kAbKeys; ++i) {
            const float4 z0 = *reinterpret_cast<const float4*>(sdZt + i * kAbST + 8 * hq);
            const float4 z1 = *reinterpret_cast<const float4*>(sdZt + i * kAbST + 8 * hq + 4);
            const float zz[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
            for (int j = 0; j < kAbMaxPairs; ++j) {
                const int pj = cl + 64 * j;
                if (pj < pairs) {
                    const float2 v = ld_f2(kvb + i * SQ + 2 * pj);
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        acc_dq[a][j].x = fmaf(zz[a], v.x, acc_dq[a][j].x);
                        acc_dq[a][j].y = fmaf(zz[a], v.y, acc_dq[a][j].y);
                    }
                }
            }
        }

        // D: dkv[s_i, :] += sum_h dz[h, i] q[h, :] + [value columns] sum_h p[h, i] dO[h, :],
        //    keys 8*hq + 4*pass .. +3 (a warp shares them), column pairs cl + 64*j
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int i0 = 8 * hq + 4 * pass;
            if (ib[i0] < 0 && ib[i0 + 1] < 0 && ib[i0 + 2] < 0 && ib[i0 + 3] < 0) continue;
            float2 acc[4][kAbMaxPairs];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int j = 0; j < kAbMaxPairs; ++j) acc[a][j] = make_float2(0.f, 0.f);
            for (int h = 0; h < hn; ++h) {
                const float4 z = *reinterpret_cast<const float4*>(sdZ + h * kAbSP + i0);
                const float4 pp = *reinterpret_cast<const float4*>(sP + h * kAbSP + i0);
                const float zz[4] = {z.x, z.y, z.z, z.w};
                const float pv[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                for (int j = 0; j < kAbMaxPairs; ++j) {
                    const int pj = cl + 64 * j;
                    if (pj < pairs) {
                        const float2 x = ld_f2(sq + h * SQ + 2 * pj);
                        float2 g = make_float2(0.f, 0.f);
                        if (pj < vpairs) g = ld_f2(sdo + h * SO + 2 * pj);
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                            acc[a][j].x = fmaf(zz[a], x.x, fmaf(pv[a], g.x, acc[a][j].x));
                            acc[a][j].y = fmaf(zz[a], x.y, fmaf(pv[a], g.y, acc[a][j].y));
                        }
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int s = ib[i0 + a];
                if (s < 0) continue;
                float* drow = dkv + (ri.key_base + s) * d_qk;
#pragma unroll
                for (int j = 0; j < kAbMaxPairs; ++j) {
                    const int pj = cl + 64 * j;
                    if (pj < pairs) atomicAdd(reinterpret_cast<float2*>(drow + 2 * pj), acc[a][j]);
                }
            }
        }
        __syncthreads();   // buffer `buf` and the p / dz tiles are reused by the next blocks
    }

#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int h = 8 * hq + a;
        if (h >= hn) continue;
        float* drow = dq + (qrow + h) * d_qk;
#pragma unroll
        for (int j = 0; j < kAbMaxPairs; ++j) {
            const int pj = cl + 64 * j;
            if (pj < pairs) *reinterpret_cast<float2*>(drow + 2 * pj) = acc_dq[a][j];
        }
    }
}

// dst[0 .. n) = 0 (n a multiple of 4, dst 16-byte aligned)
__global__ void zero_f32_kernel(float* __restrict__ dst, long long n) {
    const long long n4 = n >> 2;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        reinterpret_cast<float4*>(dst)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace dsa
