// indexer_bwd.cuh -- backward of the Lightning Indexer's scores at listed positions.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the index score of a
// query and a previous key is  I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j,:] . k_I[s,:]).
// For a gradient g on I at the positions s_m listed for row t:
//
//   dw[t,j]    = sum_m g_m * ReLU(S[j,m]),      S[j,m] = q_I[t,j,:] . k_I[s_m,:]
//   G[j,m]     = g_m * w[t,j] * [S[j,m] > 0]
//   dq_I[t,j]  = sum_m G[j,m] k_I[s_m,:]
//   dk_I[s_m] += sum_j G[j,m] q_I[t,j,:]
//
// The ReLU's decision is taken on the fp32 dot product this kernel computes.
// One CTA per query row, on the CUDA cores in fp32: the row's query heads stay
// in shared memory, the listed key rows stream through a double-buffered tile of
// 32 rows; dk_I is accumulated with fp32 atomic adds.
#pragma once

#include "attn_bwd.cuh"

namespace dsa {

constexpr int kIbThreads = 256;
constexpr int kIbHeads = 64;     // maximum indexer heads
constexpr int kIbMaxDim = 128;   // maximum indexer head dimension
constexpr int kIbKeys = 32;      // listed positions per block
constexpr int kIbSP = kIbKeys + 4;
constexpr int kIbST = kIbHeads + 4;

template <typename T>
struct IbSmem {
    int sq;
    size_t q, k, s, g, gt, w, dw, gs, idx, bytes;
    __host__ __device__ explicit IbSmem(int d) {
        sq = ab_stride<T>(d);
        q = 0;
        k = q + sizeof(T) * kIbHeads * sq;
        s = k + sizeof(T) * 2 * kIbKeys * sq;
        g = s + sizeof(float) * kIbHeads * kIbSP;
        gt = g + sizeof(float) * kIbHeads * kIbSP;
        w = gt + sizeof(float) * kIbKeys * kIbST;
        dw = w + sizeof(float) * kIbHeads;
        gs = dw + sizeof(float) * kIbHeads;       // 2 x kIbKeys score gradients
        idx = gs + sizeof(float) * 2 * kIbKeys;   // 2 x kIbKeys positions
        bytes = idx + sizeof(int) * 2 * kIbKeys;
    }
};

template <typename T>
__global__ void __launch_bounds__(kIbThreads, 1)
index_scores_bwd_kernel(RowSpec rs, const T* __restrict__ q_idx, const float* __restrict__ w,
                        const T* __restrict__ k_idx, const int* __restrict__ idx, const float* __restrict__ dsc, int k,
                        int HI, int DI, float* __restrict__ dq, float* __restrict__ dw, float* __restrict__ dk,
                        int total_q) {
    extern __shared__ __align__(16) unsigned char smem[];
    const IbSmem<T> L(DI);
    T* sq = reinterpret_cast<T*>(smem + L.q);
    T* sk = reinterpret_cast<T*>(smem + L.k);
    float* sS = reinterpret_cast<float*>(smem + L.s);
    float* sG = reinterpret_cast<float*>(smem + L.g);
    float* sGt = reinterpret_cast<float*>(smem + L.gt);
    float* sw = reinterpret_cast<float*>(smem + L.w);
    float* sdw = reinterpret_cast<float*>(smem + L.dw);
    float* sg = reinterpret_cast<float*>(smem + L.gs);
    int* sidx = reinterpret_cast<int*>(smem + L.idx);
    const int SQ = L.sq;

    const int tid = threadIdx.x, lane = tid & 31;
    const int r = total_q - 1 - static_cast<int>(blockIdx.x);
    const int pairs = DI >> 1;
    const RowInfo ri = row_info(rs, r);
    if (!ri.ok) {
        for (int e = tid; e < HI * DI; e += kIbThreads) dq[static_cast<long long>(r) * HI * DI + e] = 0.f;
        for (int e = tid; e < HI; e += kIbThreads) dw[static_cast<long long>(r) * HI + e] = 0.f;
        return;
    }
    const int n = ri.n;

    const int cpr = DI * static_cast<int>(sizeof(T)) / 16;
    constexpr int kPer = 16 / sizeof(T);
    auto load_block = [&](int b, int buf) {
        T* dst = sk + buf * kIbKeys * SQ;
        for (int c = tid; c < kIbKeys * cpr; c += kIbThreads) {
            const int i = c / cpr, part = c - i * cpr;
            const int e = b * kIbKeys + i;
            const long long ge = static_cast<long long>(r) * k + e;
            const int s = e < k ? __ldg(idx + ge) : -1;
            const bool valid = s >= 0 && s < n;
            if (part == 0) {
                if (!valid && s != -1) raise_error(DSA_ERR_DEVICE_DATA);
                sidx[buf * kIbKeys + i] = valid ? s : -1;
                sg[buf * kIbKeys + i] = valid ? __ldg(dsc + ge) : 0.f;
            }
            T* d16 = dst + i * SQ + part * kPer;
            if (valid)
                cp_async_16(smem_u32(d16), k_idx + (ri.key_base + s) * DI + part * kPer);
            else
                *reinterpret_cast<uint4*>(d16) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    ab_load_rows(sq, SQ, q_idx + static_cast<long long>(r) * HI * DI, DI, DI, kIbHeads, HI, tid);
    for (int j = tid; j < kIbHeads; j += kIbThreads) {
        sw[j] = j < HI ? __ldg(w + static_cast<long long>(r) * HI + j) : 0.f;
        sdw[j] = 0.f;
    }
    load_block(0, 0);
    cp_async_commit();

    // C's accumulators: heads 8*jq .. 8*jq+7, column pairs cl + 32*m
    const int jq = tid >> 5, cl = lane;
    float2 acc_dq[8][2];
#pragma unroll
    for (int a = 0; a < 8; ++a) acc_dq[a][0] = acc_dq[a][1] = make_float2(0.f, 0.f);

    const int nb = (k + kIbKeys - 1) / kIbKeys;
    for (int b = 0; b < nb; ++b) {
        const int buf = b & 1;
        if (b + 1 < nb) load_block(b + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        if (!__syncthreads_or(tid < kIbKeys && sidx[buf * kIbKeys + tid] >= 0)) continue;
        const T* kb = sk + buf * kIbKeys * SQ;
        const int* ib = sidx + buf * kIbKeys;
        const float* gb = sg + buf * kIbKeys;

        // A: S[j, i] for heads jb + 8*a and key ki (one key per thread)
        {
            const int jb = tid & 7, ki = tid >> 3;
            float acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = 0.f;
            for (int c = 0; c < DI; c += 2) {
                const float2 kk = ld_f2(kb + ki * SQ + c);
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const float2 x = ld_f2(sq + (jb + 8 * a) * SQ + c);
                    acc[a] = fmaf(x.x, kk.x, fmaf(x.y, kk.y, acc[a]));
                }
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) sS[(jb + 8 * a) * kIbSP + ki] = acc[a];
        }
        __syncthreads();

        // B: G = g * w * [S > 0] in both layouts; dw += sum_i g_i ReLU(S) (a warp per head)
        for (int e = tid; e < kIbHeads * kIbKeys; e += kIbThreads) {
            const int j = e / kIbKeys, i = e - j * kIbKeys;   // i = lane
            const float s = sS[j * kIbSP + i];
            const float g = gb[i];                           // 0 for an empty entry
            const float G = s > 0.f ? g * sw[j] : 0.f;
            sG[j * kIbSP + i] = G;
            sGt[i * kIbST + j] = G;
            float part = g * fmaxf(s, 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (i == 0) sdw[j] += part;
        }
        __syncthreads();

        // C: dq[j, :] += sum_i G[j, i] k[i, :]
        for (int i = 0; i < kIbKeys; ++i) {
            const float4 g0 = *reinterpret_cast<const float4*>(sGt + i * kIbST + 8 * jq);
            const float4 g1 = *reinterpret_cast<const float4*>(sGt + i * kIbST + 8 * jq + 4);
            const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int pj = cl + 32 * m;
                if (pj < pairs) {
                    const float2 v = ld_f2(kb + i * SQ + 2 * pj);
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        acc_dq[a][m].x = fmaf(gg[a], v.x, acc_dq[a][m].x);
                        acc_dq[a][m].y = fmaf(gg[a], v.y, acc_dq[a][m].y);
                    }
                }
            }
        }

        // D: dk[s_i, :] += sum_j G[j, i] q[j, :] for keys 4*jq .. 4*jq+3 (a warp shares them)
        {
            const int i0 = 4 * jq;
            if (ib[i0] >= 0 || ib[i0 + 1] >= 0 || ib[i0 + 2] >= 0 || ib[i0 + 3] >= 0) {
                float2 acc[4][2];
#pragma unroll
                for (int a = 0; a < 4; ++a) acc[a][0] = acc[a][1] = make_float2(0.f, 0.f);
                for (int j = 0; j < HI; ++j) {
                    const float4 g4 = *reinterpret_cast<const float4*>(sG + j * kIbSP + i0);
                    const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int pj = cl + 32 * m;
                        if (pj < pairs) {
                            const float2 x = ld_f2(sq + j * SQ + 2 * pj);
#pragma unroll
                            for (int a = 0; a < 4; ++a) {
                                acc[a][m].x = fmaf(gg[a], x.x, acc[a][m].x);
                                acc[a][m].y = fmaf(gg[a], x.y, acc[a][m].y);
                            }
                        }
                    }
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    const int s = ib[i0 + a];
                    if (s < 0) continue;
                    float* drow = dk + (ri.key_base + s) * DI;
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int pj = cl + 32 * m;
                        if (pj < pairs) atomicAdd(reinterpret_cast<float2*>(drow + 2 * pj), acc[a][m]);
                    }
                }
            }
        }
        __syncthreads();
    }

    const long long qrow = static_cast<long long>(r) * HI;
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int j = 8 * jq + a;
        if (j >= HI) continue;
        float* drow = dq + (qrow + j) * DI;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int pj = cl + 32 * m;
            if (pj < pairs) *reinterpret_cast<float2*>(drow + 2 * pj) = acc_dq[a][m];
        }
    }
    __syncthreads();
    for (int j = tid; j < HI; j += kIbThreads) dw[qrow + j] = sdw[j];
}

}  // namespace dsa
