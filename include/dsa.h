/*
 * dsa.h -- C ABI of libdsa: the DeepSeek Sparse Attention (DSA) forward step
 * on one NVIDIA B300 (sm_103a).
 *
 * What is computed (transformers model documentation, "DeepSeek-V3.2" page,
 * section "DeepSeek Sparse Attention (DSA)"; sizes from its DeepseekV32Config
 * parameters):
 *
 *   1. Lightning Indexer.  A light module with n_idx_heads (index_n_heads)
 *      heads of width idx_dim (index_head_dim) scores each query t against
 *      every key s at or before it, over a single-head indexer key cache:
 *          I[t,s] = sum_j w[t,j] * max(0, q_idx[t,j,:] . k_idx[s,:]),  s <= t.
 *      (The pages give the ingredients; this exact form, with no extra
 *      scale, is the reading used throughout.)
 *   2. Fine-grained token selection.  For each query keep the topk
 *      (index_topk) highest-scoring positions; when t+1 <= topk every
 *      position 0..t is kept.  Equal scores go to the lower position;
 *      -0.0 equals +0.0.
 *   3. Main MLA attention over the selected positions only, in the absorbed
 *      latent form: each of n_heads heads has a d_qk-wide query (latent
 *      kv_lora_rank + rope qk_rope_head_dim: 512 + 64); all heads share the
 *      d_qk-wide key row kv[s,:] and the value is its first d_v columns.
 *      This equals the pages' additive-mask formulation (0 on selected
 *      positions, -inf elsewhere) because exp(-inf) = 0.
 *          z[h,i] = softmax_scale * q[t,h,:] . kv[s_i,:]
 *          out[t,h,:] = sum_i softmax(z[h,:])_i kv[s_i, 0:d_v]
 *          lse[t,h]   = log sum_i exp(z[h,i])          (natural log)
 *   Each layer runs its own indexer (no state is kept between calls).
 *
 * Conventions common to every entry point
 *   - Memory: every pointer argument is DEVICE memory owned by the caller,
 *     except `const dsa_params*` (host).  The library allocates nothing;
 *     scratch for the fused calls is the caller's `workspace`.
 *   - Streams: work is enqueued asynchronously on `stream` (a cudaStream_t;
 *     NULL = legacy default stream).  Nothing synchronises the host.
 *   - Layout: row-major, last dimension contiguous, no padding except where
 *     a leading dimension (`ld`) is passed.  Tensor base addresses must be
 *     16-byte aligned.
 *   - Types: q_idx, k_idx, q, kv, caches and out have the element type
 *     `params->dtype` (DSA_BF16 or DSA_FP32); w, scores and lse are float32;
 *     cu_seqlens, cache_seqlens and selected indices are int32.
 *   - Packed ("varlen") batches: sequence b owns rows cu_seqlens[b] ..
 *     cu_seqlens[b+1]-1 of every per-token tensor; cu_seqlens[0] = 0,
 *     non-decreasing, cu_seqlens[batch] = total_q.  Positions are
 *     sequence-local and each sequence is causal on its own.  A single
 *     sequence is batch = 1, cu_seqlens = {0, L}.
 *   - Selected indices are sequence-local positions in ascending order,
 *     padded with -1 to topk entries (the DeepSeek-V4 page's marker for an
 *     empty indexer slot).
 *   - Errors: every call returns DSA_OK (0) or a negative status and never
 *     aborts the process.  Argument errors are detected on the host before
 *     anything is enqueued.  Errors that can only be seen on the device
 *     (non-monotone cu_seqlens, cache_seqlens outside [1, max_ctx], a
 *     bounded wait that ran out) make the kernels skip the affected work and
 *     raise a device error word that dsa_get_device_error() reports.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DSA_OK               0
#define DSA_ERR_ARG         -1  /* null pointer, non-positive size, bad dtype */
#define DSA_ERR_SHAPE       -2  /* inconsistent sizes (ld < max_seqlen, ...)  */
#define DSA_ERR_UNSUPPORTED -3  /* a size outside the supported limits        */
#define DSA_ERR_CUDA        -4  /* a CUDA runtime call failed                 */
#define DSA_ERR_TIMEOUT     -5  /* a bounded device-side wait ran out         */
#define DSA_ERR_WORKSPACE   -6  /* workspace pointer null or too small        */
#define DSA_ERR_DEVICE_DATA -7  /* device-side check of cu_seqlens / cache_seqlens failed */

/* element types */
#define DSA_BF16 0
#define DSA_FP32 1

/* Problem description (host struct, read during the call only).
 * DeepSeek-V3.2 values: n_idx_heads 64, idx_dim 128, n_heads 128,
 * d_qk 576, d_v 512, topk 2048, softmax_scale 1/sqrt(192), DSA_BF16. */
typedef struct dsa_params {
    int   n_idx_heads;    /* H_I: indexer heads (index_n_heads)              */
    int   idx_dim;        /* D_I: indexer head width (index_head_dim)        */
    int   n_heads;        /* H: attention heads (num_attention_heads)        */
    int   d_qk;           /* query/key width: latent + rope                  */
    int   d_v;            /* value width: the latent (kv_lora_rank), <= d_qk */
    int   topk;           /* k: tokens kept per query (index_topk)           */
    float softmax_scale;  /* multiplies q.kv before the softmax              */
    int   dtype;          /* DSA_BF16 or DSA_FP32                            */
    int   indexer_fp8;    /* 0: step 1 in dtype; 1: step 1 in its FP8 form   */
                          /* (dsa_forward only; see dsa_indexer_quantize_fp8) */
} dsa_params;

/* Limits: 1 <= n_idx_heads <= 128, 8 <= idx_dim <= 256 (multiple of 8),
 * 1 <= n_heads <= 256, 8 <= d_v <= d_qk <= 1024 (multiples of 8),
 * 1 <= topk <= 16384, max_seqlen / max_ctx <= 1048576.
 * The tensor-core path is taken for the DeepSeek-V3.2 shape in bf16
 * (64, 128, 128, 576, 512), at every batch size; other shapes run the
 * general kernels. */

/* Human-readable name of a status code (static string). */
const char* dsa_status_string(int status);

/* Bytes of `workspace` that dsa_forward needs: the fp32 index-score rows
 * (total_q x round_up(max_seqlen, 4)) plus, when the caller passes no
 * idx_out, the selected-index rows (total_q x topk int32), each 256-byte
 * aligned.  Returns 0 for invalid arguments. */
size_t dsa_workspace_size(const dsa_params* params, int total_q, int max_seqlen, int batch);

/* Bytes of `workspace` that dsa_forward_decode needs (score rows of
 * batch x round_up(max_ctx, 4) floats, plus index rows when idx_out is
 * NULL).  Returns 0 for invalid arguments. */
size_t dsa_decode_workspace_size(const dsa_params* params, int batch, int max_ctx);

/* Step 1 (Lightning Indexer) over a packed batch.
 *   q_idx  [total_q, n_idx_heads, idx_dim]   dtype
 *   w      [total_q, n_idx_heads]            float32
 *   k_idx  [total_q, idx_dim]                dtype (indexer key cache)
 *   cu_seqlens [batch+1]                     int32 (device)
 *   scores [total_q, ld] float32, written for s <= t only (row r holds the
 *          scores of the query at global row r against positions 0..t of
 *          its sequence); entries s > t are left untouched.
 *   ld >= max_seqlen, ld a multiple of 4; max_seqlen >= every length. */
int dsa_index_scores(const dsa_params* params, const void* q_idx, const float* w,
                     const void* k_idx, const int* cu_seqlens, int batch, int total_q,
                     int max_seqlen, float* scores, long long ld, void* stream);

/* Step 2 (top-k) over score rows laid out as dsa_index_scores writes them.
 * Row r (position t in its sequence) selects among scores[r*ld + 0..t].
 *   idx [total_q, topk] int32: ascending positions, -1 padded.
 * Bit-exact: the same score array always gives the same indices. */
int dsa_topk(const dsa_params* params, const float* scores, long long ld,
             const int* cu_seqlens, int batch, int total_q, int max_seqlen,
             int* idx, void* stream);

/* Step 3 (sparse MLA attention) over given selections.
 *   q   [total_q, n_heads, d_qk]  dtype
 *   kv  [total_q, d_qk]           dtype (latent + rope key rows)
 *   idx [total_q, topk]           int32, sequence-local, ascending, -1 padded;
 *                                 entry i valid iff i < min(topk, t+1)
 *   out [total_q, n_heads, d_v]   dtype
 *   lse [total_q, n_heads]        float32, or NULL */
int dsa_sparse_mla_attn(const dsa_params* params, const void* q, const void* kv,
                        const int* idx, const int* cu_seqlens, int batch, int total_q,
                        int max_seqlen, void* out, float* lse, void* stream);

/* Steps 1-3 fused over a packed prefill batch.  Arguments as above;
 * idx_out [total_q, topk] may be NULL (then the indices live in workspace).
 * workspace: device memory of at least dsa_workspace_size(...) bytes,
 * 256-byte aligned, not used concurrently by another call. */
int dsa_forward(const dsa_params* params, const void* q_idx, const float* w,
                const void* k_idx, const void* q, const void* kv,
                const int* cu_seqlens, int batch, int total_q, int max_seqlen,
                void* out, float* lse, int* idx_out,
                void* workspace, size_t workspace_bytes, void* stream);

/* Steps 1-3 for one new query per sequence over its caches (decode).
 *   q_idx [batch, n_idx_heads, idx_dim], w [batch, n_idx_heads],
 *   q [batch, n_heads, d_qk]
 *   idx_cache [batch, max_ctx, idx_dim]   indexer key cache, dtype
 *   kv_cache  [batch, max_ctx, d_qk]      latent + rope cache, dtype
 *   cache_seqlens [batch] int32 (device): valid cache length INCLUDING the
 *          new token (the caches are updated first); the query sits at
 *          position cache_seqlens[b]-1 and every cached position is a
 *          candidate.  1 <= cache_seqlens[b] <= max_ctx.
 *   out [batch, n_heads, d_v], lse [batch, n_heads] or NULL,
 *   idx_out [batch, topk] or NULL (cache positions, -1 padded). */
int dsa_forward_decode(const dsa_params* params, const void* q_idx, const float* w,
                       const void* q, const void* idx_cache, const void* kv_cache,
                       const int* cache_seqlens, int batch, int max_ctx,
                       void* out, float* lse, int* idx_out,
                       void* workspace, size_t workspace_bytes, void* stream);

/* The three steps of dsa_forward_decode as separate calls (same kernels),
 * for callers that time or replace one step.  Decode form of the arguments:
 * row b of q_idx / w / q / scores / idx / out / lse is sequence b, whose
 * query sits at cache position cache_seqlens[b]-1 and sees cache positions
 * 0 .. cache_seqlens[b]-1 (all of them candidates).
 *   dsa_index_scores_decode:  scores [batch, ld] float32 (ld >= max_ctx, a
 *       multiple of 4), entries past cache_seqlens[b]-1 left untouched.
 *   dsa_topk_decode:  idx [batch, topk] int32, cache positions ascending,
 *       -1 padded; bit-exact like dsa_topk.
 *   dsa_sparse_mla_attn_decode:  attention of q [batch, n_heads, d_qk] over
 *       the kv_cache rows idx selects; out [batch, n_heads, d_v], lse or NULL.
 * Cache layouts, limits and errors as for dsa_forward_decode. */
int dsa_index_scores_decode(const dsa_params* params, const void* q_idx, const float* w,
                            const void* idx_cache, const int* cache_seqlens, int batch,
                            int max_ctx, float* scores, long long ld, void* stream);
int dsa_topk_decode(const dsa_params* params, const float* scores, long long ld,
                    const int* cache_seqlens, int batch, int max_ctx, int* idx, void* stream);
int dsa_sparse_mla_attn_decode(const dsa_params* params, const void* q, const void* kv_cache,
                               const int* idx, const int* cache_seqlens, int batch, int max_ctx,
                               void* out, float* lse, void* stream);

/* Step 1 in its FP8 form (DeepSeek-V3.2 page, DSA section, Lightning
 * Indexer paragraph: the reference indexer runs in FP8 after a Hadamard
 * transform, which is orthogonal, Hq . Hk = q . k).  Reading used: every
 * 128-d indexer query head and key is rotated by H / sqrt(128) (Sylvester
 * order) and quantised to E4M3 (largest value 448, round to nearest even,
 * saturating) with its own scale s = amax / 448 (1 for an all-zero vector);
 *     I[t,s] = sum_j w[t,j] * ReLU(s_q[t,j] * s_k[s] * (q8[t,j,:] . k8[s,:])).
 * Supported for dtype DSA_BF16, idx_dim 128 and n_idx_heads 64.
 *
 * dsa_indexer_quantize_fp8: rotates and quantises n_vec vectors
 *   x [n_vec, 128] bf16 -> codes [n_vec, 128] (one E4M3 byte each);
 *   out [n_vec] float32 receives s, or w[i] * s when w [n_vec] is given
 *   (query heads: pass q_idx as [T*64, 128] and w as [T*64]).
 * dsa_index_scores_fp8: scores from codes, laid out as dsa_index_scores
 *   writes them: q8 [total_q, 64, 128] and wq = w * s_q [total_q, 64] from
 *   the queries, k8 [total_q, 128] and ksc = s_k [total_q] from the keys.
 * dsa_index_scores_fp8_decode: the decode form over an FP8 key cache
 *   k8_cache [batch, max_ctx, 128] with scales ksc_cache [batch, max_ctx].
 * With params->indexer_fp8 = 1, dsa_forward runs these (its workspace then
 * also holds q8, wq, k8 and ksc: dsa_workspace_size includes them); the
 * decode calls return DSA_ERR_UNSUPPORTED for that flag. */
int dsa_indexer_quantize_fp8(const dsa_params* params, const void* x, long long n_vec,
                             const float* w, void* codes, float* out, void* stream);
int dsa_index_scores_fp8(const dsa_params* params, const void* q8, const float* wq,
                         const void* k8, const float* ksc, const int* cu_seqlens, int batch,
                         int total_q, int max_seqlen, float* scores, long long ld, void* stream);
int dsa_index_scores_fp8_decode(const dsa_params* params, const void* q8, const float* wq,
                                const void* k8_cache, const float* ksc_cache,
                                const int* cache_seqlens, int batch, int max_ctx,
                                float* scores, long long ld, void* stream);

/* ---- Upstream of the path: the indexer's inputs and its key-cache update ----
 * DeepSeek-V3.2 page, "DeepSeek Sparse Attention (DSA)": the indexer scores
 * queries taken from the MLA query latent q_latent = q_a_layernorm(q_a_proj(x))
 * through its projection wq_b (sized by q_lora_rank), weights its heads with the
 * weights_proj module, and keeps its own single-head key cache of index_head_dim
 * per token, updated through update_indexer().  The page gives no further form,
 * so every projection is a bias-free linear map.
 *
 * dsa_gemm_bf16: C[m, n] = A[m, k] . B[n, k]^T on the tensor cores, bf16
 *   operands with k contiguous (rows lda / ldb elements apart), fp32
 *   accumulation, C [m, n] (rows ldc apart) written as c_dtype (DSA_BF16 rounds
 *   to nearest even, DSA_FP32 as accumulated).  Device pointers, 16-byte
 *   aligned; lda, ldb multiples of 8; ldc a multiple of 8 (bf16) or 4 (fp32).
 *   Errors: DSA_ERR_ARG (null pointer, a size < 1, bad c_dtype), DSA_ERR_SHAPE
 *   (a leading dimension too small or misaligned, a misaligned pointer),
 *   DSA_ERR_UNSUPPORTED (m > 65535 * 128).
 * dsa_indexer_inputs: for T = total_q tokens (bf16 params only),
 *   q_idx [T, H_I, D_I] = q_latent [T, q_lora_rank] . wq_b^T  (wq_b [H_I*D_I, q_lora_rank]),
 *   k_idx [T, D_I]      = x [T, hidden] . wk^T              (wk [D_I, hidden]),
 *   w [T, H_I] (fp32)   = x . w_proj^T                      (w_proj [H_I, hidden]),
 *   the inputs dsa_index_scores and dsa_forward read.  All bf16 except w;
 *   q_lora_rank, hidden, D_I multiples of 8, H_I a multiple of 4.  total_q = 0
 *   does nothing.  Errors: those of dsa_gemm_bf16, DSA_ERR_UNSUPPORTED for an
 *   fp32 params.
 * dsa_update_indexer: the decode step's append.  For every sequence b the new
 *   token's indexer key k_new [batch, D_I] and latent row kv_new [batch, d_qk]
 *   (params->dtype) are written at position cache_seqlens[b] of idx_cache
 *   [batch, max_ctx, D_I] and kv_cache [batch, max_ctx, d_qk], then
 *   cache_seqlens[b] (device memory, read and written by the call) grows by
 *   one.  A sequence whose cache is full (cache_seqlens[b] >= max_ctx) or whose
 *   length is negative is left untouched and raises DSA_ERR_DEVICE_DATA in the
 *   device error word.  Rows must be multiples of 16 bytes and the arrays
 *   16-byte aligned (DSA_ERR_SHAPE / DSA_ERR_ARG otherwise).  The caches are
 *   the dense layout the decode calls read. */
/* Paged ("dynamic") caches.  The indexer key cache and the latent cache are
 * pools of num_pages pages of page_size positions (idx_pool [num_pages *
 * page_size, D_I], kv_pool [num_pages * page_size, d_qk]); position s of
 * sequence b sits in page block_table[b * max_pages + s / page_size] (device
 * int32 [batch, max_pages]) at offset s % page_size.  page_size is a power of
 * two in [128, 2^20] (a 128-key indexer tile never crosses a page), num_pages *
 * page_size <= 2^31 - 1, max_pages * page_size <= 2^20.  A page index outside
 * [0, num_pages) raises DSA_ERR_DEVICE_DATA: the decode reads page 0 in its
 * place, and the append writes nothing for that sequence.
 * dsa_forward_decode_paged: dsa_forward_decode over paged caches, with
 *   max_ctx = max_pages * page_size (the score rows, the workspace size of
 *   dsa_decode_workspace_size(params, batch, max_ctx) and the selected
 *   positions are in that logical position space).  Same results as
 *   dsa_forward_decode over the dense caches the pages stand for.
 * dsa_update_indexer_paged: dsa_update_indexer into paged caches. */
int dsa_forward_decode_paged(const dsa_params* params, const void* q_idx, const float* w,
                             const void* q, const void* idx_pool, const void* kv_pool,
                             int num_pages, int page_size, const int* block_table, int max_pages,
                             const int* cache_seqlens, int batch, void* out, float* lse,
                             int* idx_out, void* workspace, size_t workspace_bytes, void* stream);
int dsa_update_indexer_paged(const dsa_params* params, const void* k_new, const void* kv_new,
                             int batch, int* cache_seqlens, void* idx_pool, void* kv_pool,
                             int num_pages, int page_size, const int* block_table, int max_pages,
                             void* stream);
int dsa_gemm_bf16(const void* a, long long lda, const void* b, long long ldb, int m, int n, int k,
                  void* c, long long ldc, int c_dtype, void* stream);
int dsa_indexer_inputs(const dsa_params* params, const void* q_latent, const void* x,
                       const void* wq_b, const void* wk, const void* w_proj, int total_q,
                       int q_lora_rank, int hidden, void* q_idx, void* k_idx, float* w,
                       void* stream);
int dsa_update_indexer(const dsa_params* params, const void* k_new, const void* kv_new, int batch,
                       int max_ctx, int* cache_seqlens, void* idx_cache, void* kv_cache,
                       void* stream);

/* ---- Backward (training): gradients with the selection held fixed ----
 * DeepSeek-V3.2 page, overview: DSA is a trainable sparse attention.  The
 * top-k selection is piecewise constant in the scores, so no gradient passes
 * through it; the differentiable parts are the attention over the selected
 * positions and the index scores themselves.  The pages give no loss, so the
 * gradients of the outputs are inputs.  The attention backward runs its
 * contractions on warp-level bf16 tensor-core MMAs (fp32 accumulation; p and dz
 * rounded to bf16 as operands) at the DeepSeek-V3.2 shape in bf16 and in fp32
 * on the CUDA cores otherwise; the index backward runs on the CUDA cores in
 * fp32.  Both accumulate the key-side gradients with fp32 atomic adds (so their
 * summation order, and the last bits, vary from run to run), and write fp32
 * gradients.  Packed prefill batches only (cu_seqlens as in the forward).
 *
 * dsa_sparse_mla_attn_bwd: backward of dsa_sparse_mla_attn for the same idx.
 *   q, kv, idx, cu_seqlens as in the forward; out [total_q, n_heads, d_v] and
 *   lse [total_q, n_heads] (required) are the forward's outputs for them;
 *   dout [total_q, n_heads, d_v] (dtype) the output gradient; dlse
 *   [total_q, n_heads] fp32 the lse gradient, or NULL for none.  Writes
 *     dq  [total_q, n_heads, d_qk] fp32 = scale * sum_i dz[h,i] kv[s_i,:]
 *     dkv [total_q, d_qk] fp32 (overwritten) = sum over the queries that
 *         selected row s of scale * sum_h dz[h,i] q[h,:], plus
 *         sum_h p[h,i] dO[h,:] on the first d_v columns,
 *   where p = exp(scale q.kv - lse) and dz = p (dO.kv[:d_v] - dO.O + dlse).
 *   Entries of idx outside [0, t] other than -1 are skipped and raise
 *   DSA_ERR_DEVICE_DATA; positions must be distinct, as in the forward.
 *   d_qk <= 640 and the CTA's shared tiles within 227 KB, else
 *   DSA_ERR_UNSUPPORTED.  All pointers 16-byte aligned device memory.
 * dsa_index_scores_bwd: backward of dsa_index_scores read at listed positions.
 *   q_idx, w, k_idx as in dsa_index_scores; idx [total_q, topk] int32
 *   sequence-local positions (-1 = empty; topk = params->topk per row, e.g.
 *   the selection, or every position 0..t for the whole causal row) and
 *   d_scores [total_q, topk] fp32 the gradient at each listed position.  Writes
 *     dq_idx [total_q, n_idx_heads, idx_dim] fp32, dw [total_q, n_idx_heads]
 *     fp32, dk_idx [total_q, idx_dim] fp32 (overwritten),
 *   with G[j,m] = d_scores[m] * w[j] * [q_idx[j].k_idx[s_m] > 0] (the ReLU's
 *   decision taken on the fp32 dot product): dw[j] = sum_m d_scores[m] *
 *   ReLU(q_idx[j].k_idx[s_m]), dq_idx[j] = sum_m G[j,m] k_idx[s_m],
 *   dk_idx[s] = sum over (row, m) listing s of sum_j G[j,m] q_idx[j].
 *   n_idx_heads <= 64 and idx_dim <= 128, else DSA_ERR_UNSUPPORTED.  Bad
 *   positions as above.  All pointers 16-byte aligned device memory. */
int dsa_sparse_mla_attn_bwd(const dsa_params* params, const void* q, const void* kv,
                            const int* idx, const int* cu_seqlens, int batch, int total_q,
                            int max_seqlen, const void* out, const float* lse, const void* dout,
                            const float* dlse, float* dq, float* dkv, void* stream);
int dsa_index_scores_bwd(const dsa_params* params, const void* q_idx, const float* w,
                         const void* k_idx, const int* idx, const float* d_scores,
                         const int* cu_seqlens, int batch, int total_q, int max_seqlen,
                         float* dq_idx, float* dw, float* dk_idx, void* stream);

/* Synchronises `stream`, then returns and clears the device error word:
 * DSA_OK, DSA_ERR_TIMEOUT or DSA_ERR_DEVICE_DATA (DSA_ERR_CUDA if the
 * synchronisation itself failed). */
int dsa_get_device_error(void* stream);

/* Upper bound, in nanoseconds, of every spin-wait inside the kernels
 * (default 2e9).  After it runs out a kernel raises DSA_ERR_TIMEOUT in the
 * device error word and returns instead of hanging.  Returns the previous
 * value.  Values < 1000 are clamped to 1000. */
long long dsa_set_wait_timeout_ns(long long ns);

/* Self-test of the bounded-wait path: enqueues a one-block kernel that
 * waits on an mbarrier no thread ever arrives at, with a timeout of
 * `timeout_ns`.  A correct library returns DSA_OK from this call and
 * DSA_ERR_TIMEOUT from the next dsa_get_device_error(stream). */
int dsa_selftest_wait_timeout(long long timeout_ns, void* stream);

/* Name of the kernel family a call with these parameters runs:
 * "tcgen05" (sm_103a tensor-core kernels) or "simt" (general kernels).
 * The tensor-core kernels take exactly the DeepSeek-V3.2 shape in bf16: 64
 * indexer heads of 128, 128 attention heads, query/key width 576, value
 * width 512, any index_topk, any batch and lengths.  Every other valid shape
 * (other head counts or widths, and fp32 in any shape, such as the 4 x 32 /
 * 8-head / 80 / 64 fp32 test configuration) runs the general CUDA-core
 * kernels, which compute the same definitions in fp32 arithmetic.  The FP8
 * indexer, the input projections and the paged instances of the decode
 * kernels exist for the tensor-core shape only (the CUDA-core kernels read
 * paged caches too).  "invalid" for parameters the library rejects. */
const char* dsa_path_name(const dsa_params* params);

/* Decode forward for callers that cannot allocate device memory.
 *
 * The pages describe no such call: this is a library convenience.  Some
 * callers have no way to obtain a workspace: plug-in code that runs inside
 * another framework without access to its allocator, or a serving loop
 * whose device memory is entirely owned by a pool it does not control and
 * which cannot afford the device-wide synchronisation a cudaMalloc may
 * cause in the middle of a step.  This entry point computes exactly what
 * dsa_forward_decode computes, with the same kernels and arguments, but
 * keeps its scratch (score rows and, when idx_out is NULL, the selected
 * indices) in one array of DSA_NOALLOC_SCRATCH_BYTES that the library
 * reserves statically on every GPU that loads it, for the life of the
 * process.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   Limits: batch * round_up(max_ctx, 4) <= DSA_NOALLOC_MAX_SCORES floats and,
 *   when idx_out is NULL, batch * topk <= DSA_NOALLOC_MAX_INDICES ints;
 *   larger problems return DSA_ERR_UNSUPPORTED before anything is enqueued.
 *   Set-up: the first call on a device (with that device current) looks up
 *   the array's device address and keeps it for the life of the process;
 *   make that first call before any stream capture begins.  The kept
 *   address does not survive a reset of the device (cudaDeviceReset, or the
 *   primary context being destroyed and created again): after one, the
 *   library must be unloaded and loaded again before this call is used.
 *   Sharing: every call on a device uses the same array and leaves the last
 *   call's contents in it; nothing in it has to start at zero (each call
 *   writes every entry it later reads).  Calls whose GPU work overlaps in
 *   time (different streams, or different host threads) race on the array:
 *   serialise them, for instance on one stream.
 *   Arguments, layouts and the other errors are those of dsa_forward_decode. */
#define DSA_NOALLOC_MAX_SCORES  (4u << 20)    /* 4 Mi floats: 16 MiB of score rows */
#define DSA_NOALLOC_MAX_INDICES (128u << 10)  /* 128 Ki ints: 512 KiB of indices   */
#define DSA_NOALLOC_SCRATCH_BYTES (4u * DSA_NOALLOC_MAX_SCORES + 4u * DSA_NOALLOC_MAX_INDICES)
int dsa_forward_decode_noalloc(const dsa_params* params, const void* q_idx, const float* w,
                               const void* q, const void* idx_cache, const void* kv_cache,
                               const int* cache_seqlens, int batch, int max_ctx,
                               void* out, float* lse, int* idx_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif  /* DSA_H_ */
