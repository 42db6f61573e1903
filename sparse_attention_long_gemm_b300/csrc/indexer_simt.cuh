// indexer_simt.cuh -- Lightning Indexer scores on the CUDA cores (any shape).
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", Lightning Indexer:
// I[t,s] = sum_j w[t,j] * max(0, q_I[t,j,:] . k_I[s,:]) for s <= t.
// This is the general-shape kernel (e.g. 4 heads x 32, fp32); the
// DeepSeek-V3.2 shape in bf16 runs on the tensor cores (indexer_tc.cuh).
// One CTA per query row; keys are staged 32 at a time in shared memory,
// warp w accumulates heads j = w, w+8, ... for key `lane`, and the eight
// partial sums are added in a fixed order.
#pragma once

#include "rows.cuh"

namespace dsa {

constexpr int kIdxSimtThreads = 256;
constexpr int kIdxSimtKeys = 32;

inline size_t indexer_simt_smem(int H_I, int D_I) {
    return sizeof(float) * (static_cast<size_t>(H_I) * D_I + H_I + kIdxSimtKeys * (D_I + 1) + 8 * kIdxSimtKeys);
}

template <typename T>
__global__ void __launch_bounds__(kIdxSimtThreads)
indexer_simt_kernel(RowSpec rs, const T* __restrict__ q_idx, const float* __restrict__ w,
                    const T* __restrict__ k_idx, int H_I, int D_I, float* __restrict__ scores, long long ld) {
    extern __shared__ float sm[];
    float* sq = sm;                                  // [H_I][D_I]
    float* sw = sq + H_I * D_I;                      // [H_I]
    float* sk = sw + H_I;                            // [32][D_I+1]
    float* spart = sk + kIdxSimtKeys * (D_I + 1);    // [8][32]

    const int r = blockIdx.x;
    const RowInfo ri = row_info(rs, r);
    if (!ri.ok) return;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int n = ri.n;

    const T* qr = q_idx + static_cast<long long>(r) * H_I * D_I;
    for (int i = tid; i < H_I * D_I; i += kIdxSimtThreads) sq[i] = to_f32(qr[i]);
    for (int j = tid; j < H_I; j += kIdxSimtThreads) sw[j] = w[static_cast<long long>(r) * H_I + j];

    float* srow = scores + static_cast<long long>(r) * ld;
    for (int s0 = 0; s0 < n; s0 += kIdxSimtKeys) {
        __syncthreads();
        for (int i = tid; i < kIdxSimtKeys * D_I; i += kIdxSimtThreads) {
            const int kk = i / D_I, d = i - kk * D_I;
            const int s = s0 + kk;
            sk[kk * (D_I + 1) + d] = (s < n) ? to_f32(k_idx[key_row(rs, r, ri.key_base, s) * D_I + d]) : 0.f;
        }
        __syncthreads();
        float acc = 0.f;
        const float* kr = sk + lane * (D_I + 1);
        for (int j = wid; j < H_I; j += 8) {
            const float* qj = sq + j * D_I;
            float dot = 0.f;
            for (int d = 0; d < D_I; ++d) dot = fmaf(qj[d], kr[d], dot);
            acc = fmaf(sw[j], fmaxf(dot, 0.f), acc);
        }
        spart[wid * kIdxSimtKeys + lane] = acc;
        __syncthreads();
        if (wid == 0) {
            float tot = 0.f;
#pragma unroll
            for (int v = 0; v < 8; ++v) tot += spart[v * kIdxSimtKeys + lane];
            const int s = s0 + lane;
            if (s < n) srow[s] = tot;
        }
    }
}

}  // namespace dsa
