// indexer_bwd_mma.cuh -- backward of the index scores on the tensor cores
// (DeepSeek-V3.2 indexer: 64 heads of 128, bf16).
//
// The same gradients as index_scores_bwd_kernel (see indexer_bwd.cuh), with the
// three contractions of a block of 32 listed keys on warp-level bf16 MMAs
// (m16n8k16, fp32 accumulate), operands fed by ldmatrix:
//   A  S     = q_I . k_I^T      [64 heads x 32 keys], K = 128
//   B  G     = g * w * [S > 0] (rounded to bf16), dw += sum_i g_i ReLU(S) in fp32
//   C  dq_I += G . k_I          [64 heads x 128],    K = 32 keys (registers)
//   D  dk_I  = G^T . q_I        [32 keys x 128],     K = 64 heads, fp32 atomics
// One CTA per query row; the listed key rows of the next block are gathered by
// cp.async while the current block is processed.
#pragma once

#include "attn_bwd_mma.cuh"

namespace dsa {

namespace ibm {
constexpr int kHeads = 64, kDim = 128, kKeys = 32, kThreads = 256;
constexpr int SQ = 136;         // bf16 row stride of the q_I and k_I tiles (272 B: 17 x 16 B)
constexpr int SF = kKeys + 4;   // fp32 row stride of the S tile
constexpr int SB = kKeys + 8;   // bf16 row stride of the G tile (80 B)
constexpr size_t OFF_Q = 0;
constexpr size_t OFF_K = OFF_Q + 2ull * kHeads * SQ;
constexpr size_t OFF_S = OFF_K + 2ull * 2 * kKeys * SQ;
constexpr size_t OFF_G = OFF_S + 4ull * kHeads * SF;
constexpr size_t OFF_W = OFF_G + 2ull * kHeads * SB;
constexpr size_t OFF_DW = OFF_W + 4ull * kHeads;
constexpr size_t OFF_GS = OFF_DW + 4ull * kHeads;       // score gradients of three blocks
constexpr size_t OFF_IDX = OFF_GS + 4ull * 3 * kKeys;   // positions of three blocks
constexpr size_t SMEM = OFF_IDX + 4ull * 3 * kKeys;
}  // namespace ibm

__global__ void __launch_bounds__(ibm::kThreads, 2)
index_scores_bwd_mma_kernel(RowSpec rs, const __nv_bfloat16* __restrict__ q_idx, const float* __restrict__ w,
                            const __nv_bfloat16* __restrict__ k_idx, const int* __restrict__ idx,
                            const float* __restrict__ dsc, int k, float* __restrict__ dq, float* __restrict__ dw,
                            float* __restrict__ dk, int total_q) {
    using namespace ibm;
    using bf16 = __nv_bfloat16;
    extern __shared__ __align__(16) unsigned char smem[];
    bf16* sq = reinterpret_cast<bf16*>(smem + OFF_Q);
    bf16* sk = reinterpret_cast<bf16*>(smem + OFF_K);
    float* sS = reinterpret_cast<float*>(smem + OFF_S);
    bf16* sG = reinterpret_cast<bf16*>(smem + OFF_G);
    float* sw = reinterpret_cast<float*>(smem + OFF_W);
    float* sdw = reinterpret_cast<float*>(smem + OFF_DW);
    float* sg = reinterpret_cast<float*>(smem + OFF_GS);
    int* sidx = reinterpret_cast<int*>(smem + OFF_IDX);

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int r = total_q - 1 - static_cast<int>(blockIdx.x);
    const long long qrow = static_cast<long long>(r) * kHeads;
    const RowInfo ri = row_info(rs, r);
    if (!ri.ok) {
        for (int e = tid; e < kHeads * kDim; e += kThreads) dq[qrow * kDim + e] = 0.f;
        for (int e = tid; e < kHeads; e += kThreads) dw[qrow + e] = 0.f;
        return;
    }
    const int n = ri.n;

    // positions and score gradients of block b -> slot b % 3 (warp 0, two blocks ahead)
    auto load_idx = [&](int b) {
        const int e = b * kKeys + lane;
        const long long ge = static_cast<long long>(r) * k + e;
        const int s = e < k ? __ldg(idx + ge) : -1;
        const bool valid = s >= 0 && s < n;
        if (!valid && s != -1) raise_error(DSA_ERR_DEVICE_DATA);
        sidx[(b % 3) * kKeys + lane] = valid ? s : -1;
        sg[(b % 3) * kKeys + lane] = valid ? __ldg(dsc + ge) : 0.f;
    };
    constexpr int kCpr = kDim * 2 / 16;   // 16 chunks of 16 bytes per key row
    auto load_block = [&](int b, int buf) {
        bf16* dst = sk + buf * kKeys * SQ;
        const int* ix = sidx + (b % 3) * kKeys;
        for (int c = tid; c < kKeys * kCpr; c += kThreads) {
            const int i = c / kCpr, part = c - i * kCpr;
            const int s = ix[i];
            bf16* d16 = dst + i * SQ + part * 8;
            if (s >= 0)
                cp_async_16(smem_u32(d16), k_idx + (ri.key_base + s) * kDim + part * 8);
            else
                *reinterpret_cast<uint4*>(d16) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    const int nb = (k + kKeys - 1) / kKeys;
    if (wid == 0) {
        load_idx(0);
        if (nb > 1) load_idx(1);
    }
    for (int j = tid; j < kHeads; j += kThreads) {
        sw[j] = __ldg(w + qrow + j);
        sdw[j] = 0.f;
    }
    ab_load_rows(sq, SQ, q_idx + qrow * kDim, kDim, kDim, kHeads, kHeads, tid);
    __syncthreads();
    load_block(0, 0);
    cp_async_commit();

    const uint32_t lrow = (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t lcol = 8 * (lane >> 4);
    // C's accumulators: heads 16*(wid & 3) .., columns 64*(wid >> 2) .. (8 n-tiles)
    const int cm = wid & 3, cn = wid >> 2;
    float acc_dq[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc_dq[j][0] = acc_dq[j][1] = acc_dq[j][2] = acc_dq[j][3] = 0.f;

    for (int b = 0; b < nb; ++b) {
        const int buf = b & 1;
        if (b + 1 < nb) load_block(b + 1, buf ^ 1);
        cp_async_commit();
        if (wid == 0 && b + 2 < nb) load_idx(b + 2);   // slot (b + 2) % 3 last served block b - 1
        cp_async_wait<1>();
        const int* ib = sidx + (b % 3) * kKeys;
        const float* gb = sg + (b % 3) * kKeys;
        if (!__syncthreads_or(tid < kKeys && ib[tid] >= 0)) continue;
        const uint32_t k_s = smem_u32(sk + buf * kKeys * SQ);

        // A: S, each warp a 16 x 16 tile (heads 16*(wid & 3), keys 16*(wid >> 2)); K = 128
        {
            const int nh = wid >> 2;
            float acc[2][2][4];
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int j = 0; j < 2; ++j) acc[x][j][0] = acc[x][j][1] = acc[x][j][2] = acc[x][j][3] = 0.f;
            const uint32_t a_addr = smem_u32(sq) + 2u * ((16 * cm + lrow) * SQ + lcol);
            const uint32_t b_addr =
                k_s + 2u * ((16 * nh + (lane & 7) + 8 * (lane >> 4)) * SQ + 8 * ((lane >> 3) & 1));
#pragma unroll
            for (int kk = 0; kk < kDim / 16; kk += 2) {
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    uint32_t a[4], bb[4];
                    ldsm_x4(a_addr + 32u * (kk + x), a);
                    ldsm_x4(b_addr + 32u * (kk + x), bb);
                    mma_bf16(acc[x][0], a, bb[0], bb[1]);
                    mma_bf16(acc[x][1], a, bb[2], bb[3]);
                }
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = 16 * nh + 8 * j + 2 * t4;
                *reinterpret_cast<float2*>(sS + (16 * cm + g8) * SF + col) =
                    make_float2(acc[0][j][0] + acc[1][j][0], acc[0][j][1] + acc[1][j][1]);
                *reinterpret_cast<float2*>(sS + (16 * cm + g8 + 8) * SF + col) =
                    make_float2(acc[0][j][2] + acc[1][j][2], acc[0][j][3] + acc[1][j][3]);
            }
        }
        __syncthreads();

        // B: G = g * w * [S > 0] (bf16 for C and D); dw += sum_i g_i ReLU(S) (a warp per head)
        for (int e = tid; e < kHeads * kKeys; e += kThreads) {
            const int j = e / kKeys, i = e - j * kKeys;   // i = lane
            const float s = sS[j * SF + i];
            const float gi = gb[i];                       // 0 for an empty entry
            sG[j * SB + i] = __float2bfloat16_rn(s > 0.f ? gi * sw[j] : 0.f);
            float part = gi * fmaxf(s, 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (i == 0) sdw[j] += part;
        }
        __syncthreads();

        // C: dq_I[heads 16*cm.., columns 64*cn..] += G . k_I  (K = 32 keys, k rows are K)
        {
            const uint32_t a_addr = smem_u32(sG) + 2u * ((16 * cm + lrow) * SB + lcol);
            const uint32_t b_addr = k_s + 2u * (lrow * SQ + 64 * cn + lcol);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a[4];
                ldsm_x4(a_addr + 32u * ks, a);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    uint32_t bb[4];
                    ldsm_x4_t(b_addr + 2u * (16 * ks * SQ + 16 * jj), bb);
                    mma_bf16(acc_dq[2 * jj], a, bb[0], bb[1]);
                    mma_bf16(acc_dq[2 * jj + 1], a, bb[2], bb[3]);
                }
            }
        }

        // D: dk_I[keys 16*(wid & 1).., columns 32*(wid >> 1)..] = G^T . q_I  (K = 64 heads)
        {
            const int dm = wid & 1, dn = wid >> 1;
            const int k0 = ib[16 * dm + g8], k1 = ib[16 * dm + g8 + 8];
            if (__any_sync(0xffffffffu, (k0 >= 0) || (k1 >= 0))) {
                float acc[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
                const uint32_t at_off =
                    2u * (((lane & 7) + 8 * (lane >> 4)) * SB + 16 * dm + 8 * ((lane >> 3) & 1));
#pragma unroll
                for (int ks = 0; ks < kHeads / 16; ++ks) {
                    uint32_t a[4];
                    ldsm_x4_t(smem_u32(sG) + at_off + 2u * (16 * ks * SB), a);
                    const uint32_t b_addr = smem_u32(sq) + 2u * ((16 * ks + lrow) * SQ + 32 * dn + lcol);
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        uint32_t bb[4];
                        ldsm_x4_t(b_addr + 32u * jj, bb);
                        mma_bf16(acc[2 * jj], a, bb[0], bb[1]);
                        mma_bf16(acc[2 * jj + 1], a, bb[2], bb[3]);
                    }
                }
                // lanes t4, t4^1 swap halves: four columns of one key row each, one 16-byte atomic
                const bool ev = (t4 & 1) == 0;
                const int kr = ev ? k0 : k1;
                float* drow = kr >= 0 ? dk + (ri.key_base + kr) * kDim + 32 * dn + 2 * (t4 & 2) : nullptr;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float x0 = __shfl_xor_sync(0xffffffffu, ev ? acc[j][2] : acc[j][0], 1);
                    const float x1 = __shfl_xor_sync(0xffffffffu, ev ? acc[j][3] : acc[j][1], 1);
                    const float4 v =
                        ev ? make_float4(acc[j][0], acc[j][1], x0, x1) : make_float4(x0, x1, acc[j][2], acc[j][3]);
                    if (drow != nullptr) atomicAdd(reinterpret_cast<float4*>(drow + 8 * j), v);
                }
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int col = 64 * cn + 8 * j + 2 * t4;
        *reinterpret_cast<float2*>(dq + (qrow + 16 * cm + g8) * kDim + col) = make_float2(acc_dq[j][0], acc_dq[j][1]);
        *reinterpret_cast<float2*>(dq + (qrow + 16 * cm + g8 + 8) * kDim + col) =
            make_float2(acc_dq[j][2], acc_dq[j][3]);
    }
    for (int j = tid; j < kHeads; j += kThreads) dw[qrow + j] = sdw[j];
}

}  // namespace dsa
