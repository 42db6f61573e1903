// attn_simt.cuh -- sparse MLA attention on the CUDA cores (any shape).
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the main MLA
// attention runs over the selected tokens only (the additive-mask
// formulation with exp(-inf) = 0).  Absorbed latent form: one shared
// d_qk-wide key row per position, value = its first d_v columns.
// General-shape kernel (e.g. 8 heads, 80/64, fp32).  One CTA per
// (query row, head): logits of all selected positions, an exact softmax in
// fp32, then the weighted sum of the value rows.
#pragma once

#include "rows.cuh"

namespace dsa {

constexpr int kAttnSimtThreads = 128;

inline size_t attn_simt_smem(int d_qk, int k) { return sizeof(float) * (static_cast<size_t>(d_qk) + 2 * k + 64); }

template <typename T>
__global__ void __launch_bounds__(kAttnSimtThreads)
attn_simt_kernel(RowSpec rs, const T* __restrict__ q, const T* __restrict__ kv, const int* __restrict__ idx, int k,
                 int H, int d_qk, int d_v, float scale, T* __restrict__ out, float* __restrict__ lse) {
    extern __shared__ float sm[];
    float* sq = sm;                   // [d_qk]
    float* sz = sq + d_qk;            // [k] logits, then probabilities
    int* sidx = reinterpret_cast<int*>(sz + k);   // [k] validated positions (-1 = none)
    float* sred = reinterpret_cast<float*>(sidx + k);  // [64]

    const int r = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5;
    const RowInfo ri = row_info(rs, r);
    const int n = ri.ok ? ri.n : 0;
    T* orow = out + (static_cast<long long>(r) * H + h) * d_v;

    const T* qr = q + (static_cast<long long>(r) * H + h) * d_qk;
    for (int d = tid; d < d_qk; d += kAttnSimtThreads) sq[d] = to_f32(qr[d]);
    const int* ir = idx + static_cast<long long>(r) * k;
    for (int i = tid; i < k; i += kAttnSimtThreads) {
        const int s = ir[i];
        const bool valid = (s >= 0 && s < n);
        if (!valid && s != -1) raise_error(DSA_ERR_DEVICE_DATA);
        sidx[i] = valid ? s : -1;
    }
    __syncthreads();

    float mx = -INFINITY;
    for (int i = tid; i < k; i += kAttnSimtThreads) {
        float z = -INFINITY;
        if (sidx[i] >= 0) {
            const T* kr = kv + key_row(rs, r, ri.key_base, sidx[i]) * d_qk;
            float dot = 0.f;
            for (int d = 0; d < d_qk; ++d) dot = fmaf(sq[d], to_f32(kr[d]), dot);
            z = dot * scale;
        }
        sz[i] = z;
        mx = fmaxf(mx, z);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) sred[wid] = mx;
    __syncthreads();
    mx = sred[0];
    for (int v = 1; v < kAttnSimtThreads / 32; ++v) mx = fmaxf(mx, sred[v]);
    __syncthreads();

    float sum = 0.f;
    for (int i = tid; i < k; i += kAttnSimtThreads) {
        const float p = (sidx[i] >= 0) ? expf(sz[i] - mx) : 0.f;
        sz[i] = p;
        sum += p;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) sred[32 + wid] = sum;
    __syncthreads();
    sum = 0.f;
    for (int v = 0; v < kAttnSimtThreads / 32; ++v) sum += sred[32 + v];

    if (mx == -INFINITY) {  // no valid position: zero output, lse = -inf
        for (int c = tid; c < d_v; c += kAttnSimtThreads) orow[c] = from_f32<T>(0.f);
        if (lse != nullptr && tid == 0) lse[static_cast<long long>(r) * H + h] = -INFINITY;
        return;
    }
    const float inv = 1.f / sum;
    for (int c = tid; c < d_v; c += kAttnSimtThreads) {
        float o = 0.f;
        for (int i = 0; i < k; ++i) {
            const int s = sidx[i];
            if (s >= 0) o = fmaf(sz[i], to_f32(kv[key_row(rs, r, ri.key_base, s) * d_qk + c]), o);
        }
        orow[c] = from_f32<T>(o * inv);
    }
    if (lse != nullptr && tid == 0) lse[static_cast<long long>(r) * H + h] = mx + logf(sum);
}

}  // namespace dsa
