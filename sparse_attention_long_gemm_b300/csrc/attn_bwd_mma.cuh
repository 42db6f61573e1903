// attn_bwd_mma.cuh -- backward of the sparse MLA attention on the tensor cores
// (DeepSeek-V3.2 shape: 128 heads, d_qk 576, d_v 512, bf16).
//
// The same gradients as attn_bwd_kernel (see attn_bwd.cuh for the formulas),
// with the four contractions of a block of 32 selected keys on warp-level bf16
// MMAs (m16n8k16, fp32 accumulate), operands fed from shared memory by
// ldmatrix (.trans where the contraction runs over the stored rows):
//   A  S  = q . kv^T        [32 heads x 32 keys], K = 576   (warps 0-3)
//      dP = dO . v^T        [32 heads x 32 keys], K = 512   (warps 4-7)
//   B  p = exp(scale S - lse), dz = scale p (dP - D + dlse), both rounded to bf16
//   C  dq  += dz . kv       [32 heads x 576],  K = 32 keys   (fp32 accumulators in registers)
//   D  dkv  = dz^T . q + p^T . dO (value columns)  [32 keys x 576], K = 32 heads,
//      added to the key rows with fp32 atomics
// One CTA per (query row, group of 32 heads); the kv rows of the next block are
// gathered by cp.async while the current block is processed.
#pragma once

#include "attn_bwd.cuh"

namespace dsa {

namespace abm {
constexpr int kHeads = 32, kKeys = 32, kThreads = 256;
constexpr int kDqk = 576, kDv = 512;
constexpr int SQ = 584;          // bf16 row stride of the q and kv tiles (1168 B: 73 x 16 B)
constexpr int SO = 520;          // bf16 row stride of the dO tile (1040 B: 65 x 16 B)
constexpr int SF = kKeys + 4;    // fp32 row stride of the S and dP tiles
constexpr int SB = kKeys + 8;    // bf16 row stride of the p and dz tiles (80 B: 5 x 16 B)
constexpr int kNq = kDqk / 4;    // output columns per warp in C and D (144 = 18 n-tiles of 8)
constexpr size_t OFF_Q = 0;
constexpr size_t OFF_DO = OFF_Q + 2ull * kHeads * SQ;
constexpr size_t OFF_KV = OFF_DO + 2ull * kHeads * SO;
constexpr size_t OFF_S = OFF_KV + 2ull * 2 * kKeys * SQ;
constexpr size_t OFF_DP = OFF_S + 4ull * kHeads * SF;
constexpr size_t OFF_P = OFF_DP + 4ull * kHeads * SF;
constexpr size_t OFF_DZ = OFF_P + 2ull * kHeads * SB;
constexpr size_t OFF_VEC = OFF_DZ + 2ull * kHeads * SB;
constexpr size_t OFF_IDX = OFF_VEC + 4ull * 3 * kHeads;
constexpr size_t SMEM = OFF_IDX + 4ull * 3 * kKeys;   // positions of three blocks
}  // namespace abm

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += a . b  (m16n8k16, bf16 operands, fp32 accumulators)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(abm::kThreads, 1)
attn_bwd_mma_kernel(RowSpec rs, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
                    const int* __restrict__ idx, int k, float scale, const __nv_bfloat16* __restrict__ out,
                    const float* __restrict__ lse, const __nv_bfloat16* __restrict__ dout,
                    const float* __restrict__ dlse, float* __restrict__ dq, float* __restrict__ dkv, int total_q) {
    using namespace abm;
    using bf16 = __nv_bfloat16;
    constexpr int H = 4 * kHeads;   // 128 heads in 4 groups
    extern __shared__ __align__(16) unsigned char smem[];
    bf16* sq = reinterpret_cast<bf16*>(smem + OFF_Q);
    bf16* sdo = reinterpret_cast<bf16*>(smem + OFF_DO);
    bf16* skv = reinterpret_cast<bf16*>(smem + OFF_KV);
    float* sS = reinterpret_cast<float*>(smem + OFF_S);
    float* sdP = reinterpret_cast<float*>(smem + OFF_DP);
    bf16* sP = reinterpret_cast<bf16*>(smem + OFF_P);
    bf16* sdZ = reinterpret_cast<bf16*>(smem + OFF_DZ);
    float* sD = reinterpret_cast<float*>(smem + OFF_VEC);
    float* slse = sD + kHeads;
    float* sdl = slse + kHeads;
    int* sidx = reinterpret_cast<int*>(smem + OFF_IDX);

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int r = total_q - 1 - static_cast<int>(blockIdx.x);
    const long long qrow = static_cast<long long>(r) * H + blockIdx.y * kHeads;
    const RowInfo ri = row_info(rs, r);
    if (!ri.ok) {
        for (int e = tid; e < kHeads * kDqk; e += kThreads) dq[qrow * kDqk + e] = 0.f;
        return;
    }
    const int n = ri.n;

    // Positions of block b (validated: an entry outside [0, t] other than -1 is skipped and
    // raised) go to sidx[b % 3], loaded by warp 0 two blocks ahead of their use, so that the
    // gather of a block never waits on global loads of its indices.
    auto load_idx = [&](int b) {
        const int e = b * kKeys + lane;
        const int s = e < k ? __ldg(idx + static_cast<long long>(r) * k + e) : -1;
        const bool valid = s >= 0 && s < n;
        if (!valid && s != -1) raise_error(DSA_ERR_DEVICE_DATA);
        sidx[(b % 3) * kKeys + lane] = valid ? s : -1;
    };
    constexpr int kCpr = kDqk * 2 / 16;   // 72 chunks of 16 bytes per kv row
    auto load_block = [&](int b, int buf) {
        bf16* dst = skv + buf * kKeys * SQ;
        const int* ix = sidx + (b % 3) * kKeys;
        for (int c = tid; c < kKeys * kCpr; c += kThreads) {
            const int i = c / kCpr, part = c - i * kCpr;
            const int s = ix[i];
            bf16* d16 = dst + i * SQ + part * 8;
            if (s >= 0)
                cp_async_16(smem_u32(d16), kv + (ri.key_base + s) * kDqk + part * 8);
            else
                *reinterpret_cast<uint4*>(d16) = make_uint4(0u, 0u, 0u, 0u);
        }
    };

    const int nb = (k + kKeys - 1) / kKeys;
    if (wid == 0) {
        load_idx(0);
        if (nb > 1) load_idx(1);
    }
    ab_load_rows(sq, SQ, q + qrow * kDqk, kDqk, kDqk, kHeads, kHeads, tid);
    ab_load_rows(sdo, SO, dout + qrow * kDv, kDv, kDv, kHeads, kHeads, tid);
    __syncthreads();
    load_block(0, 0);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // D = dO . O per head (a warp per head), the forward's lse (non-finite -> p = 0), dlse
    for (int h = wid; h < kHeads; h += kThreads / 32) {
        const bf16* orow = out + (qrow + h) * kDv;
        float acc = 0.f;
        for (int c = 2 * lane; c < kDv; c += 64) {
            const float2 o = ld_f2(orow + c);
            const float2 d = ld_f2(sdo + h * SO + c);
            acc = fmaf(o.x, d.x, fmaf(o.y, d.y, acc));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            sD[h] = acc;
            const float l = __ldg(lse + qrow + h);
            slse[h] = isfinite(l) ? l : INFINITY;
            sdl[h] = dlse != nullptr ? __ldg(dlse + qrow + h) : 0.f;
        }
    }

    // warp tiles: mt = 16-row half (heads in A and C, keys in D), nq = quarter of the 576 columns
    const int mt = wid & 1, nq = wid >> 1;
    const uint32_t lrow = (lane & 7) + 8 * ((lane >> 3) & 1);   // ldmatrix row of this lane
    const uint32_t lcol = 8 * (lane >> 4);                        // ldmatrix column of this lane
    float acc_dq[18][4];
#pragma unroll
    for (int j = 0; j < 18; ++j) acc_dq[j][0] = acc_dq[j][1] = acc_dq[j][2] = acc_dq[j][3] = 0.f;

    for (int b = 0; b < nb; ++b) {
        const int buf = b & 1;
        if (b + 1 < nb) load_block(b + 1, buf ^ 1);
        cp_async_commit();
        // sidx[(b + 2) % 3] last served block b - 1, whose readers all passed its last barrier
        if (wid == 0 && b + 2 < nb) load_idx(b + 2);
        cp_async_wait<1>();
        const int* ib = sidx + (b % 3) * kKeys;
        if (!__syncthreads_or(tid < kKeys && ib[tid] >= 0)) continue;
        const bf16* kvb = skv + buf * kKeys * SQ;
        const uint32_t kv_s = smem_u32(kvb);

        // A: S (warps 0-3, K = 576 over q) and dP (warps 4-7, K = 512 over dO); each warp a
        //    16 x 16 tile: rows 16*mt.., keys 16*nh..
        {
            const bool is_s = wid < 4;
            const int nh = (wid >> 1) & 1;
            const uint32_t a_s = is_s ? smem_u32(sq) : smem_u32(sdo);
            const int as = is_s ? SQ : SO;
            const int kk_n = (is_s ? kDqk : kDv) / 16;
            float acc[2][2][4];   // [K-step parity][n-tile]: four independent accumulation chains
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int j = 0; j < 2; ++j) acc[x][j][0] = acc[x][j][1] = acc[x][j][2] = acc[x][j][3] = 0.f;
            // A rows 16*mt + lrow, column 16*kk + lcol; B (kv rows = keys, non-transposed):
            // key 16*nh + (lane & 7) + 8*(lane >> 4), channel 16*kk + 8*((lane >> 3) & 1)
            const uint32_t a_addr = a_s + 2u * ((16 * mt + lrow) * as + lcol);
            const uint32_t b_addr =
                kv_s + 2u * ((16 * nh + (lane & 7) + 8 * (lane >> 4)) * SQ + 8 * ((lane >> 3) & 1));
#pragma unroll 2
            for (int kk = 0; kk < kk_n; kk += 2) {   // kk_n (36 or 32) is even
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    uint32_t a[4], bb[4];
                    ldsm_x4(a_addr + 32u * (kk + x), a);
                    ldsm_x4(b_addr + 32u * (kk + x), bb);
                    mma_bf16(acc[x][0], a, bb[0], bb[1]);
                    mma_bf16(acc[x][1], a, bb[2], bb[3]);
                }
            }
            float* dst = is_s ? sS : sdP;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int col = 16 * nh + 8 * j + 2 * t4;
                *reinterpret_cast<float2*>(dst + (16 * mt + g) * SF + col) =
                    make_float2(acc[0][j][0] + acc[1][j][0], acc[0][j][1] + acc[1][j][1]);
                *reinterpret_cast<float2*>(dst + (16 * mt + g + 8) * SF + col) =
                    make_float2(acc[0][j][2] + acc[1][j][2], acc[0][j][3] + acc[1][j][3]);
            }
        }
        __syncthreads();

        // B: p and dz = scale * p * (dP - D + dlse), rounded to bf16 for the MMAs of C and D
        for (int e = tid; e < kHeads * kKeys; e += kThreads) {
            const int h = e / kKeys, i = e - h * kKeys;
            float p = 0.f, dz = 0.f;
            if (ib[i] >= 0) {
                p = expf(fmaf(sS[h * SF + i], scale, -slse[h]));
                dz = scale * p * (sdP[h * SF + i] - sD[h] + sdl[h]);
            }
            sP[h * SB + i] = __float2bfloat16_rn(p);
            sdZ[h * SB + i] = __float2bfloat16_rn(dz);
        }
        __syncthreads();

        // C: dq[heads 16*mt.., columns nq*144..] += dz . kv  (K = 32 keys; kv rows are K)
        {
            const uint32_t a_addr = smem_u32(sdZ) + 2u * ((16 * mt + lrow) * SB + lcol);
            const uint32_t b_addr = kv_s + 2u * (lrow * SQ + nq * kNq + lcol);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a[4];
                ldsm_x4(a_addr + 32u * ks, a);
#pragma unroll
                for (int jj = 0; jj < 9; ++jj) {
                    uint32_t bb[4];
                    ldsm_x4_t(b_addr + 2u * (16 * ks * SQ + 16 * jj), bb);
                    mma_bf16(acc_dq[2 * jj], a, bb[0], bb[1]);
                    mma_bf16(acc_dq[2 * jj + 1], a, bb[2], bb[3]);
                }
            }
        }

        // D: dkv[keys 16*mt.., columns nq*144..] = dz^T . q + p^T . dO  (K = 32 heads)
        const int k0 = ib[16 * mt + g], k1 = ib[16 * mt + g + 8];
        if (__any_sync(0xffffffffu, (k0 >= 0) || (k1 >= 0))) {
            float acc[18][4];
#pragma unroll
            for (int j = 0; j < 18; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
            // A = dz^T from the [head][key] tile, transposed: head (K) 16*ks + (lane & 7) +
            // 8*(lane >> 4), key (M) 16*mt + 8*((lane >> 3) & 1)
            const uint32_t at_off = 2u * (((lane & 7) + 8 * (lane >> 4)) * SB + 16 * mt + 8 * ((lane >> 3) & 1));
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a[4];
                ldsm_x4_t(smem_u32(sdZ) + at_off + 2u * (16 * ks * SB), a);
                const uint32_t b_addr = smem_u32(sq) + 2u * ((16 * ks + lrow) * SQ + nq * kNq + lcol);
#pragma unroll
                for (int jj = 0; jj < 9; ++jj) {
                    uint32_t bb[4];
                    ldsm_x4_t(b_addr + 32u * jj, bb);
                    mma_bf16(acc[2 * jj], a, bb[0], bb[1]);
                    mma_bf16(acc[2 * jj + 1], a, bb[2], bb[3]);
                }
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                uint32_t a[4];
                ldsm_x4_t(smem_u32(sP) + at_off + 2u * (16 * ks * SB), a);
                const uint32_t b_addr = smem_u32(sdo) + 2u * ((16 * ks + lrow) * SO + nq * kNq + lcol);
#pragma unroll
                for (int jj = 0; jj < 9; ++jj) {
                    if (nq * kNq + 16 * jj >= kDv) continue;   // value columns only
                    uint32_t bb[4];
                    ldsm_x4_t(b_addr + 32u * jj, bb);
                    mma_bf16(acc[2 * jj], a, bb[0], bb[1]);
                    mma_bf16(acc[2 * jj + 1], a, bb[2], bb[3]);
                }
            }
            // A lane holds columns 2*t4, 2*t4+1 of rows g and g+8; lanes t4 and t4^1 swap halves so
            // that the even one holds four columns of row g and the odd one four of row g+8: one
            // 16-byte atomic each.
            const bool ev = (t4 & 1) == 0;
            const int kr = ev ? k0 : k1;
            float* drow = kr >= 0 ? dkv + (ri.key_base + kr) * kDqk + nq * kNq + 2 * (t4 & 2) : nullptr;
#pragma unroll
            for (int j = 0; j < 18; ++j) {
                const float x0 = __shfl_xor_sync(0xffffffffu, ev ? acc[j][2] : acc[j][0], 1);
                const float x1 = __shfl_xor_sync(0xffffffffu, ev ? acc[j][3] : acc[j][1], 1);
                const float4 v = ev ? make_float4(acc[j][0], acc[j][1], x0, x1) : make_float4(x0, x1, acc[j][2], acc[j][3]);
                if (drow != nullptr) atomicAdd(reinterpret_cast<float4*>(drow + 8 * j), v);
            }
        }
        __syncthreads();   // buffer `buf` and the p / dz tiles are reused by the next blocks
    }

#pragma unroll
    for (int j = 0; j < 18; ++j) {
        const int col = nq * kNq + 8 * j + 2 * t4;
        *reinterpret_cast<float2*>(dq + (qrow + 16 * mt + g) * kDqk + col) = make_float2(acc_dq[j][0], acc_dq[j][1]);
        *reinterpret_cast<float2*>(dq + (qrow + 16 * mt + g + 8) * kDqk + col) =
            make_float2(acc_dq[j][2], acc_dq[j][3]);
    }
}

}  // namespace dsa
