// indexer_fp8.cuh -- the Lightning Indexer's FP8 form: Hadamard rotation and
// E4M3 quantisation of its query heads and keys.
//
// DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)", Lightning Indexer
// paragraph: the reference implementation runs the indexer in FP8 after a
// Hadamard transform (rotate_activation).  The transform is orthogonal
// (Hq . Hk = q . k), so it only spreads each vector's energy over all its
// elements before quantisation.  Reading used here (the pages give no
// quantisation details): every 128-d indexer query head and key is rotated
// by H / sqrt(128) (Sylvester order) and quantised to E4M3 (the "fn"
// variant, largest value 448, round to nearest even, saturating) with its own
// scale amax / 448 (1 for an all-zero vector).
//
// The rotation runs as a fast Walsh-Hadamard transform in registers: one warp
// per vector, lane l holding elements 4l .. 4l+3, the two in-lane butterfly
// stages and five shuffle stages.  The codes are y * 448 / amax(y) of the
// unnormalised transform y = H x (the 1 / sqrt(128) cancels), and the
// scale written is amax(y) / (448 sqrt(128)).
//
// The indexer then uses  I[t,s] = s_k[s] * sum_j (w[t,j] s_q[t,j]) ReLU(q8 . k8)
// (both scales are positive, so they commute with the ReLU): for query heads
// the kernel writes w * s_q in place of s_q.
#pragma once

#include "common.cuh"

namespace dsa {

constexpr int kFp8Threads = 256;   // 8 vectors per CTA

// Two fp32 values to two E4M3 codes (round to nearest even, saturating at
// +-448): lo in the low byte.
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// One vector in registers (lane l: elements 4l .. 4l+3) -> its codes word and scale.
__device__ __forceinline__ void fp8_rotate_quantize_one(uint2 raw, int lane, uint32_t* code, float* scale) {
    float e[4];
    {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        e[0] = __low2float(a); e[1] = __high2float(a); e[2] = __low2float(b); e[3] = __high2float(b);
    }
    // butterflies of span 1 and 2 inside the lane
    {
        const float a0 = e[0] + e[1], a1 = e[0] - e[1], a2 = e[2] + e[3], a3 = e[2] - e[3];
        e[0] = a0 + a2; e[2] = a0 - a2; e[1] = a1 + a3; e[3] = a1 - a3;
    }
    // spans 4 .. 64: partner lane l ^ m; the lower lane of a pair takes the sum
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, e[i], m);
            e[i] = upper ? (o - e[i]) : (e[i] + o);
        }
    }
    float amax = fmaxf(fmaxf(fabsf(e[0]), fabsf(e[1])), fmaxf(fabsf(e[2]), fabsf(e[3])));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const float s = amax / 448.0f;                 // scale of the unnormalised transform
    uint32_t packed = 0u;
    if (amax > 0.0f) {
        const uint32_t lo = to_e4m3x2(e[0] / s, e[1] / s), hi = to_e4m3x2(e[2] / s, e[3] / s);
        packed = lo | (hi << 16);
    }
    *code = packed;
    // scale of the rotation H / sqrt(128): amax(y) / (448 sqrt(128)); an all-zero vector gets 1
    *scale = amax > 0.0f ? s * 0.08838834764831845f : 1.0f;
}

constexpr int kFp8VecPerWarp = 4;   // vectors a warp loads ahead

// x [n_vec, 128] bf16 -> codes [n_vec, 128] E4M3 and, per vector, its scale
// (w == nullptr) or w[i] * scale (w != nullptr: query heads, w of the same
// [n_vec] layout).  Each warp takes groups of kFp8VecPerWarp consecutive
// vectors, their loads issued together.
__global__ void __launch_bounds__(kFp8Threads)
fp8_rotate_quantize_kernel(const __nv_bfloat16* __restrict__ x, long long n_vec, const float* __restrict__ w,
                           uint32_t* __restrict__ codes, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const long long nwarps = static_cast<long long>(gridDim.x) * (kFp8Threads / 32);
    for (long long v0 = (static_cast<long long>(blockIdx.x) * (kFp8Threads / 32) + (threadIdx.x >> 5)) * kFp8VecPerWarp;
         v0 < n_vec; v0 += nwarps * kFp8VecPerWarp) {   // warp-uniform
        uint2 raw[kFp8VecPerWarp];
#pragma unroll
        for (int i = 0; i < kFp8VecPerWarp; ++i)
            raw[i] = (v0 + i < n_vec) ? __ldcs(reinterpret_cast<const uint2*>(x + (v0 + i) * 128) + lane)
                                      : make_uint2(0u, 0u);
#pragma unroll
        for (int i = 0; i < kFp8VecPerWarp; ++i) {
            const long long v = v0 + i;
            if (v >= n_vec) break;   // warp-uniform
            uint32_t code;
            float sc;
            fp8_rotate_quantize_one(raw[i], lane, &code, &sc);
            codes[v * 32 + lane] = code;
            if (lane == 0) out[v] = (w != nullptr) ? __ldg(w + v) * sc : sc;
        }
    }
}

}  // namespace dsa
