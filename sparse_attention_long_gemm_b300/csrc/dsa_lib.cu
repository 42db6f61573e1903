// dsa_lib.cu -- the C ABI of libdsa (declared in include/dsa.h).
//
// Host side only: argument validation, tensor-map construction for TMA,
// choice between the tensor-core kernels (DeepSeek-V3.2 shape, bf16) and the
// general CUDA-core kernels, and asynchronous launches on the caller's
// stream.  Nothing here allocates device memory or synchronises, except
// dsa_get_device_error which is documented to synchronise.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "attn_bwd.cuh"
#include "attn_bwd_mma.cuh"
#include "attn_simt.cuh"
#include "attn_tc.cuh"
#include "gemm_tc.cuh"
#include "indexer_bwd.cuh"
#include "indexer_bwd_mma.cuh"
#include "indexer_fp8.cuh"
#include "indexer_simt.cuh"
#include "indexer_tc.cuh"
#include "topk.cuh"

using namespace dsa;

namespace {

std::atomic<long long> g_timeout_ns{2000000000LL};

// prefill indexer: 4 queries (256 MMA columns) per block, 3 key stages, 2 query buffers
constexpr int kPreNQ = 4, kPreKS = 3, kPreQB = 2, kPreKC = 32;
// decode indexer: 1 query (64 columns), 5 key stages, 2 query buffers
constexpr int kDecNQ = 1, kDecKS = 5, kDecQB = 2, kDecKC = 8;
// FP8 forms: tiles are half the bytes, so more key stages fit
constexpr int kF8PreKS = 6, kF8DecKS = 8;

// largest dynamic shared memory a CTA may ask for (227 KB)
constexpr size_t kMaxDynSmem = 232448;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline long long round_up(long long x, long long m) { return (x + m - 1) / m * m; }

bool is_tc_shape(const dsa_params* p) {
    return p->dtype == DSA_BF16 && p->n_idx_heads == kIdxHeads && p->idx_dim == kIdxDim && p->n_heads == kAttnHeads &&
           p->d_qk == kAttnDqk && p->d_v == kAttnDv;
}

int check_params(const dsa_params* p) {
    if (p == nullptr) return DSA_ERR_ARG;
    if (p->dtype != DSA_BF16 && p->dtype != DSA_FP32) return DSA_ERR_ARG;
    if (p->n_idx_heads < 1 || p->idx_dim < 1 || p->n_heads < 1 || p->d_qk < 1 || p->d_v < 1 || p->topk < 1)
        return DSA_ERR_ARG;
    if (!std::isfinite(p->softmax_scale)) return DSA_ERR_ARG;
    if (p->n_idx_heads > 128 || p->idx_dim > 256 || p->idx_dim % 8 != 0 || p->n_idx_heads * p->idx_dim > 16384)
        return DSA_ERR_UNSUPPORTED;
    if (p->n_heads > 256 || p->d_qk > 1024 || p->d_v > p->d_qk || p->d_qk % 8 != 0 || p->d_v % 8 != 0 || p->d_v < 8)
        return DSA_ERR_UNSUPPORTED;
    if (p->topk > 16384) return DSA_ERR_UNSUPPORTED;
    if (p->indexer_fp8 != 0 && p->indexer_fp8 != 1) return DSA_ERR_ARG;
    if (p->indexer_fp8 && !is_tc_shape(p)) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// The FP8 form needs 128-d bf16 indexer vectors and 64 indexer heads.
bool fp8_shape(const dsa_params* p) {
    return p->dtype == DSA_BF16 && p->idx_dim == kIdxDim && p->n_idx_heads == kIdxHeads;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DSA_OK;
    return DSA_ERR_CUDA;
}

int launch_status() { return cuda_status(cudaGetLastError()); }

struct DevInfo {
    int sm_count = 0;
    size_t max_smem = 0;   // dynamic shared memory a CTA may opt into
    bool attrs_set = false;
};
std::mutex g_mu;
DevInfo g_dev[64];

int device_info(DevInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.attrs_set) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSA_ERR_CUDA;
        cudaError_t e = cudaSuccess;
        auto set = [&](const void* fn, size_t bytes) {
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        };
        set(reinterpret_cast<const void*>(&indexer_tc_kernel<kPreNQ, kPreKS, kPreQB>), IdxTc<kPreNQ, kPreKS, kPreQB>::SMEM);
        set(reinterpret_cast<const void*>(&indexer_tc_kernel<kDecNQ, kDecKS, kDecQB>), IdxTc<kDecNQ, kDecKS, kDecQB>::SMEM);
        set(reinterpret_cast<const void*>(&indexer_tc_kernel<kPreNQ, kF8PreKS, kPreQB, true>),
            IdxTc<kPreNQ, kF8PreKS, kPreQB, true>::SMEM);
        set(reinterpret_cast<const void*>(&indexer_tc_kernel<kDecNQ, kF8DecKS, kDecQB, true>),
            IdxTc<kDecNQ, kF8DecKS, kDecQB, true>::SMEM);
        set(reinterpret_cast<const void*>(&attn_tc_kernel<false>), AttnTc::SMEM);
        set(reinterpret_cast<const void*>(&attn_tc_kernel<true>), AttnTc::SMEM);
        set(reinterpret_cast<const void*>(&indexer_tc_kernel<kDecNQ, kDecKS, kDecQB, false, true>),
            IdxTc<kDecNQ, kDecKS, kDecQB>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<64, true>), GemmTc<64>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<128, true>), GemmTc<128>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<256, true>), GemmTc<256>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<64, false>), GemmTc<64>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<128, false>), GemmTc<128>::SMEM);
        set(reinterpret_cast<const void*>(&gemm_tc_kernel<256, false>), GemmTc<256>::SMEM);
        set(reinterpret_cast<const void*>(&topk_rows_kernel), TkSmem::bytes(kTkMaxLen));
        set(reinterpret_cast<const void*>(&indexer_simt_kernel<float>), indexer_simt_smem(128, 128));
        set(reinterpret_cast<const void*>(&indexer_simt_kernel<__nv_bfloat16>), indexer_simt_smem(128, 128));
        set(reinterpret_cast<const void*>(&attn_simt_kernel<float>), attn_simt_smem(1024, 16384));
        set(reinterpret_cast<const void*>(&attn_simt_kernel<__nv_bfloat16>), attn_simt_smem(1024, 16384));
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        d.max_smem = std::min(static_cast<size_t>(optin), kMaxDynSmem);
        set(reinterpret_cast<const void*>(&attn_bwd_kernel<float>), d.max_smem);
        set(reinterpret_cast<const void*>(&attn_bwd_kernel<__nv_bfloat16>), d.max_smem);
        set(reinterpret_cast<const void*>(&attn_bwd_mma_kernel), abm::SMEM);
        set(reinterpret_cast<const void*>(&index_scores_bwd_mma_kernel), ibm::SMEM);
        set(reinterpret_cast<const void*>(&index_scores_bwd_kernel<float>), IbSmem<float>(kIbMaxDim).bytes);
        set(reinterpret_cast<const void*>(&index_scores_bwd_kernel<__nv_bfloat16>),
            IbSmem<__nv_bfloat16>(kIbMaxDim).bytes);
        if (e != cudaSuccess) return DSA_ERR_CUDA;
        d.attrs_set = true;
    }
    *out = &d;
    return DSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (row stride = cols elements), box
// [box_rows, box_cols] with the given swizzle (box_cols * 2 bytes must not
// exceed the swizzle span).
int make_tmap_bf16(CUtensorMap* tm, const void* base, long long rows, long long cols, int box_rows, int box_cols = 64,
                   CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = encode_fn();
    if (fn == nullptr) return DSA_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

// 2-D bf16 tensor [rows, cols] with rows `ld` elements apart, box [box_rows, 64], 128-byte swizzle.
int make_tmap_bf16_ld(CUtensorMap* tm, const void* base, long long rows, long long cols, long long ld, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return DSA_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

// 2-D uint8 tensor [rows, cols] (E4M3 codes), box [box_rows, 128 bytes], 128-byte swizzle.
int make_tmap_u8(CUtensorMap* tm, const void* base, long long rows, long long cols, int box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return DSA_ERR_CUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// stage launchers (arguments already validated)
// ---------------------------------------------------------------------------
// C[M, N] = A[M, K] . B[N, K]^T: a tile width that the output columns fill, one persistent CTA per SM
int run_gemm(const void* a, long long lda, const void* b, long long ldb, int m, int n, int k, void* c, long long ldc,
             bool out_bf16, cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    const int bn = n >= 256 ? 256 : (n > 64 ? 128 : 64);
    CUtensorMap ta, tb;
    if ((rc = make_tmap_bf16_ld(&ta, a, m, k, lda, kGemmBM)) != DSA_OK) return rc;
    if ((rc = make_tmap_bf16_ld(&tb, b, n, k, ldb, bn)) != DSA_OK) return rc;
    const long long ntiles = static_cast<long long>((n + bn - 1) / bn) * ((m + kGemmBM - 1) / kGemmBM);
    const unsigned long long to = static_cast<unsigned long long>(g_timeout_ns.load());
    // persistent: as many CTAs as fit on the SMs at once (narrow tiles fit two per SM, which the
    // bandwidth-bound projections need), at most one per tile
#define DSA_GEMM_LAUNCH(BN_, OB_)                                                                        \
    do {                                                                                                 \
        int per_sm = 1;                                                                                  \
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_tc_kernel<BN_, OB_>, kGemmThreads, \
                                                          GemmTc<BN_>::SMEM) != cudaSuccess || per_sm < 1) \
            per_sm = 1;                                                                                  \
        const dim3 grid(static_cast<unsigned>(std::min<long long>(ntiles, 1LL * per_sm * di->sm_count))); \
        gemm_tc_kernel<BN_, OB_><<<grid, kGemmThreads, GemmTc<BN_>::SMEM, st>>>(ta, tb, m, n, k, c, ldc, to); \
    } while (0)
    if (out_bf16) {
        if (bn == 256) DSA_GEMM_LAUNCH(256, true); else if (bn == 128) DSA_GEMM_LAUNCH(128, true); else DSA_GEMM_LAUNCH(64, true);
    } else {
        if (bn == 256) DSA_GEMM_LAUNCH(256, false); else if (bn == 128) DSA_GEMM_LAUNCH(128, false); else DSA_GEMM_LAUNCH(64, false);
    }
#undef DSA_GEMM_LAUNCH
    return launch_status();
}

int run_index_scores(const dsa_params* p, const void* q_idx, const float* w, const void* k_idx, const RowSpec& rs,
                     int rows, long long key_rows, float* scores, long long ld, cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    const unsigned long long to = static_cast<unsigned long long>(g_timeout_ns.load());
    if (is_tc_shape(p)) {
        CUtensorMap tq, tk;
        const bool dec = rs.decode != 0;
        const int bn = dec ? IdxTc<kDecNQ, kDecKS, kDecQB>::BN : IdxTc<kPreNQ, kPreKS, kPreQB>::BN;
        if ((rc = make_tmap_bf16(&tq, q_idx, static_cast<long long>(rows) * kIdxHeads, kIdxDim, bn)) != DSA_OK)
            return rc;
        if ((rc = make_tmap_bf16(&tk, k_idx, key_rows, kIdxDim, kIdxTileKeys)) != DSA_OK) return rc;
        // The kernel keeps a per-sequence work prefix in shared memory for at most kIdxTcMaxBatch
        // sequences; longer batches run as consecutive launches over chunks of sequences (prefill:
        // cu_seqlens entries hold absolute rows, so a chunk just starts further into the array;
        // decode: `base` gives the chunk's first sequence).
        for (int b0 = 0; b0 < rs.batch; b0 += kIdxTcMaxBatch) {
            RowSpec ch = rs;
            ch.lens = rs.lens + b0;
            ch.batch = std::min(kIdxTcMaxBatch, rs.batch - b0);
            ch.base = dec ? rs.base + b0 : 0;
            if (!dec) {
                using C = IdxTc<kPreNQ, kPreKS, kPreQB>;
                indexer_tc_kernel<kPreNQ, kPreKS, kPreQB>
                    <<<di->sm_count, C::THREADS, C::SMEM, st>>>(tq, tk, ch, w, nullptr, scores, ld, kPreKC, to);
            } else {
                using C = IdxTc<kDecNQ, kDecKS, kDecQB>;
                if (rs.pages != nullptr)
                    indexer_tc_kernel<kDecNQ, kDecKS, kDecQB, false, true>
                        <<<di->sm_count, C::THREADS, C::SMEM, st>>>(tq, tk, ch, w, nullptr, scores, ld, kDecKC, to);
                else
                    indexer_tc_kernel<kDecNQ, kDecKS, kDecQB>
                        <<<di->sm_count, C::THREADS, C::SMEM, st>>>(tq, tk, ch, w, nullptr, scores, ld, kDecKC, to);
            }
            if ((rc = launch_status()) != DSA_OK) return rc;
        }
        return DSA_OK;
    }
    const size_t sm = indexer_simt_smem(p->n_idx_heads, p->idx_dim);
    if (p->dtype == DSA_BF16)
        indexer_simt_kernel<__nv_bfloat16><<<rows, kIdxSimtThreads, sm, st>>>(
            rs, static_cast<const __nv_bfloat16*>(q_idx), w, static_cast<const __nv_bfloat16*>(k_idx), p->n_idx_heads,
            p->idx_dim, scores, ld);
    else
        indexer_simt_kernel<float><<<rows, kIdxSimtThreads, sm, st>>>(rs, static_cast<const float*>(q_idx), w,
                                                                      static_cast<const float*>(k_idx),
                                                                      p->n_idx_heads, p->idx_dim, scores, ld);
    return launch_status();
}

// FP8 form of step 1 from codes: q8 [rows, 64, 128] and k8 [key_rows, 128] E4M3, wq = w * s_q
// [rows, 64], ksc = s_k [key_rows].
int run_index_scores_fp8(const uint8_t* q8, const float* wq, const uint8_t* k8, const float* ksc, const RowSpec& rs,
                         int rows, long long key_rows, float* scores, long long ld, cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    const unsigned long long to = static_cast<unsigned long long>(g_timeout_ns.load());
    CUtensorMap tq, tk;
    const bool dec = rs.decode != 0;
    const int bn = dec ? IdxTc<kDecNQ, kF8DecKS, kDecQB, true>::BN : IdxTc<kPreNQ, kF8PreKS, kPreQB, true>::BN;
    if ((rc = make_tmap_u8(&tq, q8, static_cast<long long>(rows) * kIdxHeads, kIdxDim, bn)) != DSA_OK) return rc;
    if ((rc = make_tmap_u8(&tk, k8, key_rows, kIdxDim, kIdxTileKeys)) != DSA_OK) return rc;
    for (int b0 = 0; b0 < rs.batch; b0 += kIdxTcMaxBatch) {   // chunks of sequences, as for bf16
        RowSpec ch = rs;
        ch.lens = rs.lens + b0;
        ch.batch = std::min(kIdxTcMaxBatch, rs.batch - b0);
        ch.base = dec ? rs.base + b0 : 0;
        if (!dec) {
            using C = IdxTc<kPreNQ, kF8PreKS, kPreQB, true>;
            indexer_tc_kernel<kPreNQ, kF8PreKS, kPreQB, true>
                <<<di->sm_count, C::THREADS, C::SMEM, st>>>(tq, tk, ch, wq, ksc, scores, ld, kPreKC, to);
        } else {
            using C = IdxTc<kDecNQ, kF8DecKS, kDecQB, true>;
            indexer_tc_kernel<kDecNQ, kF8DecKS, kDecQB, true>
                <<<di->sm_count, C::THREADS, C::SMEM, st>>>(tq, tk, ch, wq, ksc, scores, ld, kDecKC, to);
        }
        if ((rc = launch_status()) != DSA_OK) return rc;
    }
    return DSA_OK;
}

// Rotation and E4M3 quantisation of n_vec 128-d bf16 vectors.
int run_quantize_fp8(const void* x, long long n_vec, const float* w, uint8_t* codes, float* out, cudaStream_t st) {
    if (n_vec == 0) return DSA_OK;
    DevInfo* di = nullptr;
    const int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    // enough warps for every vector group, at most 8 CTAs per SM (grid-stride beyond that)
    const long long per = (kFp8Threads / 32) * kFp8VecPerWarp;
    const long long blocks = std::min<long long>((n_vec + per - 1) / per, 8LL * di->sm_count);
    fp8_rotate_quantize_kernel<<<static_cast<unsigned>(blocks), kFp8Threads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), n_vec, w, reinterpret_cast<uint32_t*>(codes), out);
    return launch_status();
}

int run_topk(const dsa_params* p, const float* scores, long long ld, const RowSpec& rs, int rows, int* idx,
             cudaStream_t st) {
    if (rs.max_len <= kTkMaxLen) {
        DevInfo* di = nullptr;
        const int rc = device_info(&di);
        if (rc != DSA_OK) return rc;
        // persistent: as many 256-thread CTAs as fit on every SM (4 or 5: the bitmaps follow the
        // longest row)
        const int smem = TkSmem::bytes(rs.max_len);
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_rows_kernel, kTkThreads, smem) != cudaSuccess ||
            per_sm < 1) {
            per_sm = 1;
            (void)cudaGetLastError();   // a failed query only shrinks the grid
        }
        const int grid = std::max(1, std::min(rows, per_sm * di->sm_count));
        topk_rows_kernel<<<grid, kTkThreads, smem, st>>>(rs, scores, ld, p->topk, rows, idx);
    } else {
        topk_kernel<<<rows, kTopkThreads, 0, st>>>(rs, scores, ld, p->topk, idx);
    }
    return launch_status();
}

int run_attn(const dsa_params* p, const void* q, const void* kv, const int* idx, const RowSpec& rs, int rows,
             long long key_rows, void* out, float* lse, cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    if (is_tc_shape(p)) {
        CUtensorMap tq, tqr;
        const long long qrows = static_cast<long long>(rows) * kAttnHeads;
        if ((rc = make_tmap_bf16(&tq, q, qrows, kAttnDqk, kAttnHeads)) != DSA_OK) return rc;
        if ((rc = make_tmap_bf16(&tqr, q, qrows, kAttnDqk, 64, 32, CU_TENSOR_MAP_SWIZZLE_64B)) != DSA_OK) return rc;
        (void)key_rows;
        const float scale_log2 = p->softmax_scale * 1.4426950408889634f;
        const int nclusters = std::max(1, std::min(rows, di->sm_count / 2));
        const unsigned long long to = static_cast<unsigned long long>(g_timeout_ns.load());
        if (rs.pages != nullptr)
            attn_tc_kernel<true><<<2 * nclusters, kAttnThreads, AttnTc::SMEM, st>>>(
                tq, tqr, static_cast<const __nv_bfloat16*>(kv), idx, rs, rows, p->topk, scale_log2,
                static_cast<__nv_bfloat16*>(out), lse, to);
        else
            attn_tc_kernel<false><<<2 * nclusters, kAttnThreads, AttnTc::SMEM, st>>>(
                tq, tqr, static_cast<const __nv_bfloat16*>(kv), idx, rs, rows, p->topk, scale_log2,
                static_cast<__nv_bfloat16*>(out), lse, to);
        return launch_status();
    }
    const dim3 grid(rows, p->n_heads);
    const size_t sm = attn_simt_smem(p->d_qk, p->topk);
    if (p->dtype == DSA_BF16)
        attn_simt_kernel<__nv_bfloat16><<<grid, kAttnSimtThreads, sm, st>>>(
            rs, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kv), idx, p->topk,
            p->n_heads, p->d_qk, p->d_v, p->softmax_scale, static_cast<__nv_bfloat16*>(out), lse);
    else
        attn_simt_kernel<float><<<grid, kAttnSimtThreads, sm, st>>>(
            rs, static_cast<const float*>(q), static_cast<const float*>(kv), idx, p->topk, p->n_heads, p->d_qk,
            p->d_v, p->softmax_scale, static_cast<float*>(out), lse);
    return launch_status();
}

// dst[0 .. n) = 0 on the stream (n a multiple of 4)
int run_zero(float* dst, long long n, cudaStream_t st) {
    if (n <= 0) return DSA_OK;
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    const long long blocks = std::min<long long>((n / 4 + 255) / 256, 8LL * di->sm_count);
    zero_f32_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(dst, n);
    return launch_status();
}

// Backward of step 4 for packed prefill rows: dkv zeroed, then one CTA per (row, 32 heads); the
// DeepSeek-V3.2 shape in bf16 runs its contractions on the tensor cores, other shapes on the CUDA cores.
int run_attn_bwd(const dsa_params* p, const void* q, const void* kv, const int* idx, const RowSpec& rs, int rows,
                 const void* out, const float* lse, const void* dout, const float* dlse, float* dq, float* dkv,
                 cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    const size_t sm = p->dtype == DSA_BF16 ? AbSmem<__nv_bfloat16>(p->d_qk, p->d_v).bytes
                                           : AbSmem<float>(p->d_qk, p->d_v).bytes;
    if (sm > di->max_smem) return DSA_ERR_UNSUPPORTED;
    if ((rc = run_zero(dkv, static_cast<long long>(rows) * p->d_qk, st)) != DSA_OK) return rc;
    const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>((p->n_heads + kAbHeads - 1) / kAbHeads));
    if (is_tc_shape(p)) {
        using T = __nv_bfloat16;
        attn_bwd_mma_kernel<<<grid, abm::kThreads, abm::SMEM, st>>>(
            rs, static_cast<const T*>(q), static_cast<const T*>(kv), idx, p->topk, p->softmax_scale,
            static_cast<const T*>(out), lse, static_cast<const T*>(dout), dlse, dq, dkv, rows);
    } else if (p->dtype == DSA_BF16) {
        using T = __nv_bfloat16;
        attn_bwd_kernel<T><<<grid, kAbThreads, sm, st>>>(
            rs, static_cast<const T*>(q), static_cast<const T*>(kv), idx, p->topk, p->n_heads, p->d_qk, p->d_v,
            p->softmax_scale, static_cast<const T*>(out), lse, static_cast<const T*>(dout), dlse, dq, dkv, rows);
    } else {
        attn_bwd_kernel<float><<<grid, kAbThreads, sm, st>>>(
            rs, static_cast<const float*>(q), static_cast<const float*>(kv), idx, p->topk, p->n_heads, p->d_qk,
            p->d_v, p->softmax_scale, static_cast<const float*>(out), lse, static_cast<const float*>(dout), dlse, dq,
            dkv, rows);
    }
    return launch_status();
}

// Backward of step 1 at listed positions for packed prefill rows: dk zeroed, then one CTA per row;
// the DeepSeek-V3.2 indexer shape (64 x 128, bf16) runs its contractions on the tensor cores.
int run_index_scores_bwd(const dsa_params* p, const void* q_idx, const float* w, const void* k_idx, const int* idx,
                         const float* dsc, const RowSpec& rs, int rows, float* dq, float* dw, float* dk,
                         cudaStream_t st) {
    DevInfo* di = nullptr;
    int rc = device_info(&di);
    if (rc != DSA_OK) return rc;
    if ((rc = run_zero(dk, static_cast<long long>(rows) * p->idx_dim, st)) != DSA_OK) return rc;
    if (fp8_shape(p)) {
        using T = __nv_bfloat16;
        index_scores_bwd_mma_kernel<<<rows, ibm::kThreads, ibm::SMEM, st>>>(
            rs, static_cast<const T*>(q_idx), w, static_cast<const T*>(k_idx), idx, dsc, p->topk, dq, dw, dk, rows);
    } else if (p->dtype == DSA_BF16) {
        using T = __nv_bfloat16;
        index_scores_bwd_kernel<T><<<rows, kIbThreads, IbSmem<T>(p->idx_dim).bytes, st>>>(
            rs, static_cast<const T*>(q_idx), w, static_cast<const T*>(k_idx), idx, dsc, p->topk, p->n_idx_heads,
            p->idx_dim, dq, dw, dk, rows);
    } else {
        index_scores_bwd_kernel<float><<<rows, kIbThreads, IbSmem<float>(p->idx_dim).bytes, st>>>(
            rs, static_cast<const float*>(q_idx), w, static_cast<const float*>(k_idx), idx, dsc, p->topk,
            p->n_idx_heads, p->idx_dim, dq, dw, dk, rows);
    }
    return launch_status();
}

int check_prefill_common(const dsa_params* p, const int* cu, int batch, int total_q, int max_seqlen) {
    int rc = check_params(p);
    if (rc != DSA_OK) return rc;
    if (cu == nullptr || batch < 1 || total_q < 0 || max_seqlen < 1) return DSA_ERR_ARG;
    if (max_seqlen > (1 << 20)) return DSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(total_q) * p->n_heads * p->d_qk > (1LL << 40)) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// Checks shared by every decode call (sizes and the cache lengths array).
int check_decode_common(const dsa_params* p, const int* cache_seqlens, int batch, int max_ctx) {
    int rc = check_params(p);
    if (rc != DSA_OK) return rc;
    if (cache_seqlens == nullptr || batch < 1 || max_ctx < 1) return DSA_ERR_ARG;
    if (max_ctx > (1 << 20)) return DSA_ERR_UNSUPPORTED;
    if (static_cast<long long>(batch) * max_ctx > (1LL << 31) / 64) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

// Workspace bytes of the FP8 indexer's operands for T tokens: q8 [T,64,128], w * s_q [T,64],
// k8 [T,128], s_k [T], each 256-byte aligned.
long long fp8_workspace(long long T) {
    return round_up(T * kIdxHeads * kIdxDim, 256) + round_up(T * kIdxHeads * 4, 256) + round_up(T * kIdxDim, 256) +
           round_up(T * 4, 256);
}

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
    switch (status) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_ARG: return "DSA_ERR_ARG: null pointer, non-positive size or bad dtype";
        case DSA_ERR_SHAPE: return "DSA_ERR_SHAPE: inconsistent sizes";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: size outside the supported limits";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA runtime call failed";
        case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded device-side wait ran out";
        case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
        case DSA_ERR_DEVICE_DATA: return "DSA_ERR_DEVICE_DATA: cu_seqlens / cache_seqlens / indices out of range";
        default: return "unknown dsa status";
    }
}

const char* dsa_path_name(const dsa_params* params) {
    if (check_params(params) != DSA_OK) return "invalid";
    return is_tc_shape(params) ? "tcgen05" : "simt";
}

size_t dsa_workspace_size(const dsa_params* params, int total_q, int max_seqlen, int batch) {
    if (check_params(params) != DSA_OK || total_q < 0 || max_seqlen < 1 || batch < 1) return 0;
    const long long ld = round_up(max_seqlen, 4);
    const long long sc = round_up(static_cast<long long>(total_q) * ld * 4, 256);
    const long long ix = round_up(static_cast<long long>(total_q) * params->topk * 4, 256);
    return static_cast<size_t>(sc + ix + (params->indexer_fp8 ? fp8_workspace(total_q) : 0));
}

size_t dsa_decode_workspace_size(const dsa_params* params, int batch, int max_ctx) {
    if (check_params(params) != DSA_OK || batch < 1 || max_ctx < 1) return 0;
    const long long ld = round_up(max_ctx, 4);
    const long long sc = round_up(static_cast<long long>(batch) * ld * 4, 256);
    const long long ix = round_up(static_cast<long long>(batch) * params->topk * 4, 256);
    return static_cast<size_t>(sc + ix);
}

int dsa_index_scores(const dsa_params* params, const void* q_idx, const float* w, const void* k_idx,
                     const int* cu_seqlens, int batch, int total_q, int max_seqlen, float* scores, long long ld,
                     void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (q_idx == nullptr || w == nullptr || k_idx == nullptr || scores == nullptr) return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(scores)) return DSA_ERR_ARG;
    if (ld < max_seqlen || ld % 4 != 0) return DSA_ERR_SHAPE;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_index_scores(params, q_idx, w, k_idx, rs, total_q, total_q, scores, ld,
                            static_cast<cudaStream_t>(stream));
}

int dsa_topk(const dsa_params* params, const float* scores, long long ld, const int* cu_seqlens, int batch,
             int total_q, int max_seqlen, int* idx, void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (scores == nullptr || idx == nullptr) return DSA_ERR_ARG;
    if (!aligned16(scores) || !aligned16(idx)) return DSA_ERR_ARG;
    if (ld < max_seqlen || ld % 4 != 0) return DSA_ERR_SHAPE;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_topk(params, scores, ld, rs, total_q, idx, static_cast<cudaStream_t>(stream));
}

int dsa_sparse_mla_attn(const dsa_params* params, const void* q, const void* kv, const int* idx,
                        const int* cu_seqlens, int batch, int total_q, int max_seqlen, void* out, float* lse,
                        void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (q == nullptr || kv == nullptr || idx == nullptr || out == nullptr) return DSA_ERR_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)))
        return DSA_ERR_ARG;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_attn(params, q, kv, idx, rs, total_q, total_q, out, lse, static_cast<cudaStream_t>(stream));
}

int dsa_forward(const dsa_params* params, const void* q_idx, const float* w, const void* k_idx, const void* q,
                const void* kv, const int* cu_seqlens, int batch, int total_q, int max_seqlen, void* out, float* lse,
                int* idx_out, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (q_idx == nullptr || w == nullptr || k_idx == nullptr || q == nullptr || kv == nullptr || out == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(q) || !aligned16(kv) ||
        !aligned16(out) || (lse && !aligned16(lse)) || (idx_out && !aligned16(idx_out)))
        return DSA_ERR_ARG;
    if (total_q == 0) return DSA_OK;
    const size_t need = dsa_workspace_size(params, total_q, max_seqlen, batch);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DSA_ERR_WORKSPACE;
    const long long ld = round_up(max_seqlen, 4);
    float* scores = static_cast<float*>(workspace);
    int* idx = idx_out ? idx_out
                       : reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                                round_up(static_cast<long long>(total_q) * ld * 4, 256));
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (params->indexer_fp8) {
        // rotate and quantise q_I (folding s_q into w) and k_I into the workspace, then score
        char* f8 = static_cast<char*>(workspace) + round_up(static_cast<long long>(total_q) * ld * 4, 256) +
                   round_up(static_cast<long long>(total_q) * params->topk * 4, 256);
        const long long T = total_q;
        uint8_t* q8 = reinterpret_cast<uint8_t*>(f8);
        float* wq = reinterpret_cast<float*>(f8 + round_up(T * kIdxHeads * kIdxDim, 256));
        uint8_t* k8 = reinterpret_cast<uint8_t*>(reinterpret_cast<char*>(wq) + round_up(T * kIdxHeads * 4, 256));
        float* ksc = reinterpret_cast<float*>(reinterpret_cast<char*>(k8) + round_up(T * kIdxDim, 256));
        if ((rc = run_quantize_fp8(q_idx, T * kIdxHeads, w, q8, wq, st)) != DSA_OK) return rc;
        if ((rc = run_quantize_fp8(k_idx, T, nullptr, k8, ksc, st)) != DSA_OK) return rc;
        if ((rc = run_index_scores_fp8(q8, wq, k8, ksc, rs, total_q, total_q, scores, ld, st)) != DSA_OK) return rc;
    } else if ((rc = run_index_scores(params, q_idx, w, k_idx, rs, total_q, total_q, scores, ld, st)) != DSA_OK) {
        return rc;
    }
    if ((rc = run_topk(params, scores, ld, rs, total_q, idx, st)) != DSA_OK) return rc;
    return run_attn(params, q, kv, idx, rs, total_q, total_q, out, lse, st);
}

int dsa_forward_decode(const dsa_params* params, const void* q_idx, const float* w, const void* q,
                       const void* idx_cache, const void* kv_cache, const int* cache_seqlens, int batch, int max_ctx,
                       void* out, float* lse, int* idx_out, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (params->indexer_fp8) return DSA_ERR_UNSUPPORTED;   // the FP8 key cache has its own stage call
    if (q_idx == nullptr || w == nullptr || q == nullptr || idx_cache == nullptr || kv_cache == nullptr ||
        out == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(q) || !aligned16(idx_cache) || !aligned16(kv_cache) ||
        !aligned16(out) || (lse && !aligned16(lse)) || (idx_out && !aligned16(idx_out)))
        return DSA_ERR_ARG;
    const size_t need = dsa_decode_workspace_size(params, batch, max_ctx);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DSA_ERR_WORKSPACE;
    const long long ld = round_up(max_ctx, 4);
    float* scores = static_cast<float*>(workspace);
    int* idx = idx_out ? idx_out
                       : reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                                round_up(static_cast<long long>(batch) * ld * 4, 256));
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long key_rows = static_cast<long long>(batch) * max_ctx;
    if ((rc = run_index_scores(params, q_idx, w, idx_cache, rs, batch, key_rows, scores, ld, st)) != DSA_OK) return rc;
    if ((rc = run_topk(params, scores, ld, rs, batch, idx, st)) != DSA_OK) return rc;
    return run_attn(params, q, kv_cache, idx, rs, batch, key_rows, out, lse, st);
}

int dsa_index_scores_decode(const dsa_params* params, const void* q_idx, const float* w, const void* idx_cache,
                            const int* cache_seqlens, int batch, int max_ctx, float* scores, long long ld,
                            void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (q_idx == nullptr || w == nullptr || idx_cache == nullptr || scores == nullptr) return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(idx_cache) || !aligned16(scores)) return DSA_ERR_ARG;
    if (ld < max_ctx || ld % 4 != 0) return DSA_ERR_SHAPE;
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    return run_index_scores(params, q_idx, w, idx_cache, rs, batch, static_cast<long long>(batch) * max_ctx, scores,
                            ld, static_cast<cudaStream_t>(stream));
}

int dsa_topk_decode(const dsa_params* params, const float* scores, long long ld, const int* cache_seqlens, int batch,
                    int max_ctx, int* idx, void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (scores == nullptr || idx == nullptr) return DSA_ERR_ARG;
    if (!aligned16(scores) || !aligned16(idx)) return DSA_ERR_ARG;
    if (ld < max_ctx || ld % 4 != 0) return DSA_ERR_SHAPE;
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    return run_topk(params, scores, ld, rs, batch, idx, static_cast<cudaStream_t>(stream));
}

int dsa_sparse_mla_attn_decode(const dsa_params* params, const void* q, const void* kv_cache, const int* idx,
                               const int* cache_seqlens, int batch, int max_ctx, void* out, float* lse,
                               void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (q == nullptr || kv_cache == nullptr || idx == nullptr || out == nullptr) return DSA_ERR_ARG;
    if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(idx) || !aligned16(out) || (lse && !aligned16(lse)))
        return DSA_ERR_ARG;
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    return run_attn(params, q, kv_cache, idx, rs, batch, static_cast<long long>(batch) * max_ctx, out, lse,
                    static_cast<cudaStream_t>(stream));
}

int dsa_indexer_quantize_fp8(const dsa_params* params, const void* x, long long n_vec, const float* w, void* codes,
                             float* out, void* stream) {
    int rc = check_params(params);
    if (rc != DSA_OK) return rc;
    if (!fp8_shape(params)) return DSA_ERR_UNSUPPORTED;
    if (x == nullptr || codes == nullptr || out == nullptr || n_vec < 0) return DSA_ERR_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(out) || (w && !aligned16(w))) return DSA_ERR_ARG;
    return run_quantize_fp8(x, n_vec, w, static_cast<uint8_t*>(codes), out, static_cast<cudaStream_t>(stream));
}

int dsa_index_scores_fp8(const dsa_params* params, const void* q8, const float* wq, const void* k8, const float* ksc,
                         const int* cu_seqlens, int batch, int total_q, int max_seqlen, float* scores, long long ld,
                         void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (!fp8_shape(params)) return DSA_ERR_UNSUPPORTED;
    if (q8 == nullptr || wq == nullptr || k8 == nullptr || ksc == nullptr || scores == nullptr) return DSA_ERR_ARG;
    if (!aligned16(q8) || !aligned16(wq) || !aligned16(k8) || !aligned16(ksc) || !aligned16(scores))
        return DSA_ERR_ARG;
    if (ld < max_seqlen || ld % 4 != 0) return DSA_ERR_SHAPE;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_index_scores_fp8(static_cast<const uint8_t*>(q8), wq, static_cast<const uint8_t*>(k8), ksc, rs, total_q,
                                total_q, scores, ld, static_cast<cudaStream_t>(stream));
}

int dsa_index_scores_fp8_decode(const dsa_params* params, const void* q8, const float* wq, const void* k8_cache,
                                const float* ksc_cache, const int* cache_seqlens, int batch, int max_ctx,
                                float* scores, long long ld, void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (!fp8_shape(params)) return DSA_ERR_UNSUPPORTED;
    if (q8 == nullptr || wq == nullptr || k8_cache == nullptr || ksc_cache == nullptr || scores == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q8) || !aligned16(wq) || !aligned16(k8_cache) || !aligned16(ksc_cache) || !aligned16(scores))
        return DSA_ERR_ARG;
    if (ld < max_ctx || ld % 4 != 0) return DSA_ERR_SHAPE;
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    return run_index_scores_fp8(static_cast<const uint8_t*>(q8), wq, static_cast<const uint8_t*>(k8_cache), ksc_cache,
                                rs, batch, static_cast<long long>(batch) * max_ctx, scores, ld,
                                static_cast<cudaStream_t>(stream));
}

int dsa_sparse_mla_attn_bwd(const dsa_params* params, const void* q, const void* kv, const int* idx,
                            const int* cu_seqlens, int batch, int total_q, int max_seqlen, const void* out,
                            const float* lse, const void* dout, const float* dlse, float* dq, float* dkv,
                            void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (q == nullptr || kv == nullptr || idx == nullptr || out == nullptr || lse == nullptr || dout == nullptr ||
        dq == nullptr || dkv == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q) || !aligned16(kv) || !aligned16(idx) || !aligned16(out) || !aligned16(lse) ||
        !aligned16(dout) || (dlse && !aligned16(dlse)) || !aligned16(dq) || !aligned16(dkv))
        return DSA_ERR_ARG;
    const size_t sm = params->dtype == DSA_BF16 ? AbSmem<__nv_bfloat16>(params->d_qk, params->d_v).bytes
                                                : AbSmem<float>(params->d_qk, params->d_v).bytes;
    if (params->d_qk > kAbMaxDqk || sm > kMaxDynSmem) return DSA_ERR_UNSUPPORTED;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_attn_bwd(params, q, kv, idx, rs, total_q, out, lse, dout, dlse, dq, dkv,
                        static_cast<cudaStream_t>(stream));
}

int dsa_index_scores_bwd(const dsa_params* params, const void* q_idx, const float* w, const void* k_idx,
                         const int* idx, const float* d_scores, const int* cu_seqlens, int batch, int total_q,
                         int max_seqlen, float* dq_idx, float* dw, float* dk_idx, void* stream) {
    int rc = check_prefill_common(params, cu_seqlens, batch, total_q, max_seqlen);
    if (rc != DSA_OK) return rc;
    if (q_idx == nullptr || w == nullptr || k_idx == nullptr || idx == nullptr || d_scores == nullptr ||
        dq_idx == nullptr || dw == nullptr || dk_idx == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(idx) || !aligned16(d_scores) ||
        !aligned16(dq_idx) || !aligned16(dw) || !aligned16(dk_idx))
        return DSA_ERR_ARG;
    if (params->n_idx_heads > kIbHeads || params->idx_dim > kIbMaxDim) return DSA_ERR_UNSUPPORTED;
    if (total_q == 0) return DSA_OK;
    const RowSpec rs{cu_seqlens, batch, 0, max_seqlen};
    return run_index_scores_bwd(params, q_idx, w, k_idx, idx, d_scores, rs, total_q, dq_idx, dw, dk_idx,
                                static_cast<cudaStream_t>(stream));
}

int dsa_get_device_error(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
    return v;
}

long long dsa_set_wait_timeout_ns(long long ns) {
    if (ns < 1000) ns = 1000;
    return g_timeout_ns.exchange(ns);
}

}  // extern "C"

namespace dsa {
// one thread waits on an mbarrier that nothing arrives at
__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        wait_bar(smem_u32(&bar), 0, timeout_ns, &abort_flag);
    }
}
}  // namespace dsa

extern "C" int dsa_selftest_wait_timeout(long long timeout_ns, void* stream) {
    if (timeout_ns < 1000) timeout_ns = 1000;
    if (timeout_ns > 10000000000LL) return DSA_ERR_ARG;
    dsa::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(timeout_ns));
    return launch_status();
}

// ---------------------------------------------------------------------------
// dsa_forward_decode_noalloc: decode forward with library-owned scratch.
//
// For callers that cannot allocate device memory (see include/dsa.h).  The
// scratch is one statically reserved array per device; host code must not
// pass the array's name to a kernel (in host code it only stands for the
// symbol), so its device address is looked up once per device with
// cudaGetSymbolAddress and cached.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device (looked up on
// the first call for that device).
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return DSA_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return DSA_OK;
}

}  // namespace

extern "C" int dsa_forward_decode_noalloc(const dsa_params* params, const void* q_idx, const float* w,
                                          const void* q, const void* idx_cache, const void* kv_cache,
                                          const int* cache_seqlens, int batch, int max_ctx, void* out,
                                          float* lse, int* idx_out, void* stream) {
    int rc = check_decode_common(params, cache_seqlens, batch, max_ctx);
    if (rc != DSA_OK) return rc;
    if (params->indexer_fp8) return DSA_ERR_UNSUPPORTED;   // the FP8 key cache has its own stage call
    if (q_idx == nullptr || w == nullptr || q == nullptr || idx_cache == nullptr || kv_cache == nullptr ||
        out == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(q) || !aligned16(idx_cache) || !aligned16(kv_cache) ||
        !aligned16(out) || (lse && !aligned16(lse)) || (idx_out && !aligned16(idx_out)))
        return DSA_ERR_ARG;
    const long long ld = round_up(max_ctx, 4);
    if (static_cast<long long>(batch) * ld > static_cast<long long>(DSA_NOALLOC_MAX_SCORES)) return DSA_ERR_UNSUPPORTED;
    if (idx_out == nullptr &&
        static_cast<long long>(batch) * params->topk > static_cast<long long>(DSA_NOALLOC_MAX_INDICES))
        return DSA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(&scratch)) != DSA_OK) return rc;
    float* scores = static_cast<float*>(scratch);
    int* idx = idx_out ? idx_out
                       : reinterpret_cast<int*>(static_cast<char*>(scratch) + 4ull * DSA_NOALLOC_MAX_SCORES);
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long key_rows = static_cast<long long>(batch) * max_ctx;
    if ((rc = run_index_scores(params, q_idx, w, idx_cache, rs, batch, key_rows, scores, ld, st)) != DSA_OK) return rc;
    if ((rc = run_topk(params, scores, ld, rs, batch, idx, st)) != DSA_OK) return rc;
    return run_attn(params, q, kv_cache, idx, rs, batch, key_rows, out, lse, st);
}

// ---------------------------------------------------------------------------
// upstream of the path: the indexer's input projections and its cache update
// ---------------------------------------------------------------------------
extern "C" int dsa_gemm_bf16(const void* a, long long lda, const void* b, long long ldb, int m, int n, int k, void* c,
                             long long ldc, int c_dtype, void* stream) {
    if (a == nullptr || b == nullptr || c == nullptr) return DSA_ERR_ARG;
    if (m < 1 || n < 1 || k < 1 || (c_dtype != DSA_BF16 && c_dtype != DSA_FP32)) return DSA_ERR_ARG;
    if (lda < k || ldb < k || ldc < n) return DSA_ERR_SHAPE;
    // TMA: 16-byte aligned bases and row strides; the epilogue's 16-byte stores likewise
    if (!aligned16(a) || !aligned16(b) || !aligned16(c) || lda % 8 != 0 || ldb % 8 != 0 ||
        ldc % (c_dtype == DSA_BF16 ? 8 : 4) != 0)
        return DSA_ERR_SHAPE;
    if (m > 65535 * kGemmBM) return DSA_ERR_UNSUPPORTED;
    return run_gemm(a, lda, b, ldb, m, n, k, c, ldc, c_dtype == DSA_BF16, static_cast<cudaStream_t>(stream));
}

extern "C" int dsa_indexer_inputs(const dsa_params* params, const void* q_latent, const void* x, const void* wq_b,
                                  const void* wk, const void* w_proj, int total_q, int q_lora_rank, int hidden,
                                  void* q_idx, void* k_idx, float* w, void* stream) {
    int rc = check_params(params);
    if (rc != DSA_OK) return rc;
    if (params->dtype != DSA_BF16) return DSA_ERR_UNSUPPORTED;
    if (total_q < 0 || q_lora_rank < 1 || hidden < 1) return DSA_ERR_ARG;
    if (total_q == 0) return DSA_OK;
    if (q_latent == nullptr || x == nullptr || wq_b == nullptr || wk == nullptr || w_proj == nullptr ||
        q_idx == nullptr || k_idx == nullptr || w == nullptr)
        return DSA_ERR_ARG;
    const int H = params->n_idx_heads, D = params->idx_dim;
    if (q_lora_rank % 8 != 0 || hidden % 8 != 0 || (H * D) % 8 != 0 || D % 8 != 0 || H % 4 != 0) return DSA_ERR_SHAPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = dsa_gemm_bf16(q_latent, q_lora_rank, wq_b, q_lora_rank, total_q, H * D, q_lora_rank, q_idx, H * D,
                            DSA_BF16, st)) != DSA_OK)
        return rc;
    if ((rc = dsa_gemm_bf16(x, hidden, wk, hidden, total_q, D, hidden, k_idx, D, DSA_BF16, st)) != DSA_OK) return rc;
    return dsa_gemm_bf16(x, hidden, w_proj, hidden, total_q, H, hidden, w, H, DSA_FP32, st);
}

namespace {
// Validates a paged cache (page pools of num_pages pages of page_size positions, block table
// [batch, max_pages]) and fills the paged fields of rs.
int paged_spec(int num_pages, int page_size, const int* block_table, int max_pages, RowSpec* rs) {
    if (block_table == nullptr || num_pages < 1 || max_pages < 1) return DSA_ERR_ARG;
    if (page_size < 128 || page_size > (1 << 20) || (page_size & (page_size - 1)) != 0) return DSA_ERR_SHAPE;
    if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
    int lg = 0;
    while ((1 << lg) < page_size) ++lg;
    rs->pages = block_table;
    rs->page_log2 = lg;
    rs->max_pages = max_pages;
    rs->num_pages = num_pages;
    return DSA_OK;
}

int update_indexer(const dsa_params* params, const void* k_new, const void* kv_new, const RowSpec& rs,
                   int* cache_seqlens, void* idx_cache, void* kv_cache, void* stream) {
    if (k_new == nullptr || kv_new == nullptr || cache_seqlens == nullptr || idx_cache == nullptr ||
        kv_cache == nullptr)
        return DSA_ERR_ARG;
    const int es = params->dtype == DSA_BF16 ? 2 : 4;
    const int kb = params->idx_dim * es, vb = params->d_qk * es;
    if (kb % 16 != 0 || vb % 16 != 0) return DSA_ERR_SHAPE;
    if (!aligned16(k_new) || !aligned16(kv_new) || !aligned16(idx_cache) || !aligned16(kv_cache)) return DSA_ERR_ARG;
    update_indexer_kernel<<<rs.batch, kUpdThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        rs, static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(kv_new), kb, vb, cache_seqlens,
        static_cast<uint8_t*>(idx_cache), static_cast<uint8_t*>(kv_cache));
    return launch_status();
}
}  // namespace

extern "C" int dsa_update_indexer(const dsa_params* params, const void* k_new, const void* kv_new, int batch,
                                  int max_ctx, int* cache_seqlens, void* idx_cache, void* kv_cache, void* stream) {
    int rc = check_params(params);
    if (rc != DSA_OK) return rc;
    if (batch < 1 || max_ctx < 1) return DSA_ERR_ARG;
    const RowSpec rs{cache_seqlens, batch, 1, max_ctx};
    return update_indexer(params, k_new, kv_new, rs, cache_seqlens, idx_cache, kv_cache, stream);
}

extern "C" int dsa_update_indexer_paged(const dsa_params* params, const void* k_new, const void* kv_new, int batch,
                                        int* cache_seqlens, void* idx_pool, void* kv_pool, int num_pages,
                                        int page_size, const int* block_table, int max_pages, void* stream) {
    int rc = check_params(params);
    if (rc != DSA_OK) return rc;
    if (batch < 1) return DSA_ERR_ARG;
    RowSpec rs{cache_seqlens, batch, 1, 0};
    if ((rc = paged_spec(num_pages, page_size, block_table, max_pages, &rs)) != DSA_OK) return rc;
    if (static_cast<long long>(max_pages) * page_size > (1 << 20)) return DSA_ERR_UNSUPPORTED;
    rs.max_len = max_pages * page_size;
    return update_indexer(params, k_new, kv_new, rs, cache_seqlens, idx_pool, kv_pool, stream);
}

extern "C" int dsa_forward_decode_paged(const dsa_params* params, const void* q_idx, const float* w, const void* q,
                                        const void* idx_pool, const void* kv_pool, int num_pages, int page_size,
                                        const int* block_table, int max_pages, const int* cache_seqlens, int batch,
                                        void* out, float* lse, int* idx_out, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (params == nullptr) return DSA_ERR_ARG;
    RowSpec rs{cache_seqlens, batch, 1, 0};
    int rc = paged_spec(num_pages, page_size, block_table, max_pages, &rs);
    if (rc != DSA_OK) return rc;
    if (static_cast<long long>(max_pages) * page_size > (1 << 20)) return DSA_ERR_UNSUPPORTED;
    const int max_ctx = max_pages * page_size;
    rs.max_len = max_ctx;
    if ((rc = check_decode_common(params, cache_seqlens, batch, max_ctx)) != DSA_OK) return rc;
    if (params->indexer_fp8) return DSA_ERR_UNSUPPORTED;
    if (q_idx == nullptr || w == nullptr || q == nullptr || idx_pool == nullptr || kv_pool == nullptr ||
        out == nullptr)
        return DSA_ERR_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(q) || !aligned16(idx_pool) || !aligned16(kv_pool) ||
        !aligned16(out) || (lse && !aligned16(lse)) || (idx_out && !aligned16(idx_out)))
        return DSA_ERR_ARG;
    const size_t need = dsa_decode_workspace_size(params, batch, max_ctx);
    if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return DSA_ERR_WORKSPACE;
    const long long ld = round_up(max_ctx, 4);
    float* scores = static_cast<float*>(workspace);
    int* idx = idx_out ? idx_out
                       : reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                                round_up(static_cast<long long>(batch) * ld * 4, 256));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long key_rows = static_cast<long long>(num_pages) * page_size;
    if ((rc = run_index_scores(params, q_idx, w, idx_pool, rs, batch, key_rows, scores, ld, st)) != DSA_OK) return rc;
    if ((rc = run_topk(params, scores, ld, rs, batch, idx, st)) != DSA_OK) return rc;
    return run_attn(params, q, kv_pool, idx, rs, batch, key_rows, out, lse, st);
}
