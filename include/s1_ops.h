/*
 * s1 — kernel-level entry points and instrumentation (libs1.so).
 *
 * These expose single steps of the decision path on DEVICE pointers so each kernel can be
 * checked on its own against an independent reference, and timed. They are blocking
 * (they synchronise the given stream before returning) and may allocate small device
 * temporaries; they are not needed by the decision API in s1.h.
 * Return codes and s1_last_error() as in s1.h.
 */
#ifndef S1_OPS_H_
#define S1_OPS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define S1_MAX_OPTIONS 1024     /* option ids per question */

/* profiling classes of s1_profile_read */
enum { S1_PROF_GEMM = 0, S1_PROF_GDN = 1, S1_PROF_ATTN = 2, S1_PROF_NORM = 3, S1_PROF_OTHER = 4,
       S1_PROF_NCLASS = 8 };

/* GEMM epilogues of s1_op_gemm */
enum { S1_EPI_F32 = 0, S1_EPI_F16 = 1, S1_EPI_RESADD = 2, S1_EPI_SWIGLU = 3 };

/* Y = epi(X[M,K] . W[N,K]^T): f16 operands (row-major, K contiguous), fp32 accumulate.
 * The projections of every decoder layer (gated delta-rule in-projection
 * [q|k|v|a|b], attention in-projection [q|k|v], out-projections, SwiGLU MLP) are of
 * this form (layer definition of the hybrid decoder; LoRA merged into W at load,
 * System1-Omni issue #10 plan item 3).
 *   S1_EPI_F32:    out fp32 [M, ldo] = acc
 *   S1_EPI_F16:    out f16 [M, ldo] = acc (round to nearest even)
 *   S1_EPI_RESADD: out fp32 [M, ldo] += acc        (residual stream)
 *   S1_EPI_SWIGLU: W rows interleaved in blocks of 16 gate rows then 16 up rows;
 *                  out f16 [M, ldo], N/2 columns: silu(gate) * up
 * impl: 0 = tcgen05 tensor-core kernel (the product path: single-CTA or CTA-pair tiles, the
 *       planner's choice), 1 = SIMT reference, 2 = tensor-core kernel restricted to CTA-pair
 *       tiles (256 x N per pair, tcgen05.mma.cta_group::2), 3 = restricted to single-CTA tiles.
 *       Any other value: S1_ERR_INVALID_ARG.
 * Requires K % 64 == 0 and N % 32 == 0 (SWIGLU: N % 32 == 0); X, W 16-byte aligned. */
int s1_op_gemm(const void* X, const void* W, int32_t M, int32_t N, int32_t K, int32_t epi,
               void* out, int32_t ldo, int32_t impl, void* stream);

/* s1_op_gemm without any device allocation. This entry point has no counterpart in the
 * pages: it exists for callers that cannot call cudaMalloc when they run a projection —
 * code whose device memory is owned and budgeted by another framework, real-time loops that
 * must not allocate (an allocation can synchronise the device), or processes whose memory is
 * fixed up front. Same arguments, plan and results as s1_op_gemm (blocking; stream may be
 * NULL). Its split-K partials and its error word live in fixed device arrays inside the
 * library: S1_NOALLOC_WS_FLOATS floats (16 MiB) plus 256 bytes, reserved on every GPU that
 * loads the library until the process exits. The first call on a device looks up the arrays'
 * device addresses (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call shares the arrays: calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller. A shape whose
 * split-K plan needs more than S1_NOALLOC_WS_FLOATS floats of partials is rejected with
 * S1_ERR_BUDGET before any device work. */
#define S1_NOALLOC_WS_FLOATS (4 * 1024 * 1024)
int s1_op_gemm_noalloc(const void* X, const void* W, int32_t M, int32_t N, int32_t K, int32_t epi,
                       void* out, int32_t ldo, void* stream);

/* The tensor-core GEMM plan the planner's heuristic picks for an M x N x K product with
 * epilogue `epi` on a GPU of num_sms SMs: pair = 0 for the single-CTA kernel family, 1 for the
 * CTA-pair family (as impl 3 / 2 of s1_op_gemm). out (host, 7 int32): tile width BN, CTAs per
 * weight tile (always 1: no load is shared across a cluster), CTA pair (0/1), K splits, 64-deep
 * k-blocks per split, 128-row M tiles, N tiles. Host logic only, callable without a GPU: the CTAs
 * (or pairs) of a tile width that fit at once come from the device's occupancy query when a
 * device is present, else one per SM (or per two SMs) (the first answer is kept for the process). The autotuner's measured choice, which can replace a
 * split-free plan on first use of a shape in a model, is not applied. Errors: INVALID_ARG
 * (M < 1, N % 32, K % 64, epi outside 0..3, num_sms < 1, NULL out). */
int s1_gemm_plan(int32_t M, int32_t N, int32_t K, int32_t epi, int32_t num_sms, int32_t pair, int32_t* out);

/* Gated delta rule over packed sequences, per head (Yang, Kautz & Hatamizadeh 2024):
 *   q, k <- L2-normalised (x / sqrt(sum x^2 + l2_eps)), alpha = exp(-softplus(a)),
 *   beta = sigmoid(b), S_t = alpha S_{t-1}(I - beta k k^T) + beta v k^T, o_t = S_t q_t.
 * proj: fp32 [R, 2*H*dk + H*dv + 2*H] rows [q | k | v | a | b] (read; the token-by-token path,
 * taken for head sizes other than 64 and 128, normalises q and k in place).
 * Sequence s covers rows row0[s] .. row0[s]+len[s]-1 (host arrays). S0: device fp32
 * [n_seq, H, dv, dk] initial states or NULL (zero). S_out: device [n_seq, H, dv, dk] final
 * states or NULL. out: f16 [R, H*dv]. */
int s1_op_gdn(float* proj, int32_t R, int32_t H, int32_t dk, int32_t dv, float l2_eps,
              int32_t n_seq, const int32_t* row0, const int32_t* len, const float* S0,
              float* S_out, void* out, void* stream);

/* Causal GQA attention with continuation (System1-Omni RFC #114 section 4, "Branching").
 * q f16 [R, Hq, hd] and k_new, v_new f16 [R, Hkv, hd] (already rotated). Sequence s
 * (rows row0[s] .. +len[s]) attends to the P cached keys kv_cache = f16 [2, P, Hkv, hd]
 * (K plane then V plane; NULL when P == 0) and causally to its own rows.
 * softmax(q.k / sqrt(hd)) v; q head h reads kv head floor(h*Hkv/Hq). out f16 [R, Hq*hd]. */
int s1_op_attention(const void* q, const void* k_new, const void* v_new, const void* kv_cache,
                    int32_t P, int32_t n_seq, const int32_t* row0, const int32_t* len, int32_t Hq,
                    int32_t Hkv, int32_t hd, void* out, void* stream);

/* out f16 [R, d] = x / sqrt(mean(x^2) + eps) * w;  x fp32 [R, d], w fp32 [d]. */
int s1_op_rmsnorm(const float* x, const float* w, int32_t R, int32_t d, float eps, void* out,
                  void* stream);

/* ---- instrumentation of a model (handles from s1.h) -------------------------------------
 * s1_profile(m, 1) starts recording CUDA events around every launch of the model on its
 * stream (class per S1_PROF_*); s1_profile_read synchronises and returns, per class, the
 * summed device milliseconds, the algorithmic flops and bytes counted, and the launch
 * count (arrays of S1_PROF_NCLASS; any may be NULL). s1_profile(m, 0) stops and clears. */
struct s1_model;
int s1_profile(struct s1_model* m, int enable);
int s1_profile_read(struct s1_model* m, double* ms, double* flops, double* bytes, long* count);
/* Cumulative counters of a model: kernels launched by its forward passes, and bytes copied
 * host->device / device->host by the blocking calls (ids, metadata, embeddings, results). */
int s1_counters(struct s1_model* m, long long* launches, long long* h2d_bytes, long long* d2h_bytes);
/* 0 = tensor-core GEMM (default), 1 = SIMT GEMM for every projection (debug only). */
int s1_set_gemm_impl(struct s1_model* m, int impl);
/* Layer trace (a debugging and verification aid, no counterpart in the pages): while set, every
 * forward pass of the model copies its fp32 residual stream into d_trace, stream-ordered —
 * plane 0 after the embedding rows, plane l + 1 after layer l — as [n_layers + 1][R][d_model]
 * in the call's packed row order (prefill: the prefix rows; decide: the questions' suffix rows
 * in question order; one sweep: every prefix, then every question's suffix). d_trace is a
 * device buffer of capacity_floats floats owned by the caller, who keeps it alive while it is
 * set; a call that needs more fails with S1_ERR_BUDGET before any launch. NULL clears it.
 * Synchronises the model's stream. */
int s1_set_layer_trace(struct s1_model* m, float* d_trace, long long capacity_floats);

#ifdef __cplusplus
}
#endif
#endif /* S1_OPS_H_ */
