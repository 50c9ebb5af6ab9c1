/*
 * s1 — prefill-only decisions on a hybrid gated-delta-rule / GQA decoder (GB300, sm_103a).
 *
 * C ABI of libs1.so. All entry points return an s1 status code (0 = S1_OK);
 * on a non-zero return, s1_last_error() gives a thread-local message.
 *
 * What the library computes (sources by page and section):
 *  - A decision is one prefill pass and a softmax over the option tokens'
 *    logits at the last position; nothing is decoded (System1-Omni issue #10,
 *    "Support Cua-S1 4B 0.2", plan item 1).
 *  - The common state prefix is encoded once; every question suffix then runs
 *    as an isolated continuation of the prefix's immutable snapshot:
 *    full-attention KV plus the FP32 gated delta-rule state (System1-Omni RFC
 *    #114, section 4 "Branching" row; section 5 "Shared-prefix execution").
 *  - Option logits are rows of the tied input embedding (RFC #114, section 3).
 *  - Answer types choice / score / noul and the two confidences are those of
 *    the sys1rust README ("Each question gets one of 3 answer types" and the
 *    confidence bullets).
 *  - LoRA adapters (rank 32, alpha 64 in the pages) are merged into the base
 *    weights once, at load (issue #10 plan item 3; RFC #114 section 1).
 *  - Inputs are validated before any device work and rejected with explicit
 *    errors; budgets are enforced (RFC #114 section 2, "Validate ... before
 *    dispatch ... Return explicit errors").
 *  - Blocking dispatch: the host-pointer calls return when results are in
 *    caller memory (RFC #114 section 2, serial scheduler with blocking dispatch);
 *    nothing is freed while device work that uses it is in flight (section 2,
 *    "Preserve resource ownership until device work finishes").
 *
 * Layouts are row-major. Weight matrices use the [out, in] convention.
 * Ownership: every input pointer is read during the call only; the caller keeps
 * it. Handles (s1_model, s1_state) are owned by the library until destroyed.
 * Thread safety: one model must not be used from two threads at once.
 */
#ifndef S1_H_
#define S1_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define S1_OK 0
#define S1_ERR_INVALID_ARG 1      /* bad id, length, option count or shape              */
#define S1_ERR_INVALID_HANDLE 2   /* NULL / destroyed / foreign model or state          */
#define S1_ERR_OOM 3              /* an allocation failed (nothing leaked)              */
#define S1_ERR_BUDGET 4           /* a declared row / question budget was exceeded      */
#define S1_ERR_CUDA 5             /* a CUDA runtime call failed                          */
#define S1_ERR_DEVICE_TIMEOUT 6   /* a bounded device-side wait gave up                  */
#define S1_ERR_UNSUPPORTED 7      /* shape the kernels do not handle (message says why)  */

enum { S1_F32 = 0, S1_BF16 = 1 };            /* dtype of the host weight arrays        */
enum { S1_CHOICE = 0, S1_SCORE = 1, S1_NOUL = 2 };

typedef struct s1_model s1_model;
typedef struct s1_state s1_state;

/* Model shape. Layer l is full attention iff layer_is_full[l] != 0, otherwise a
 * gated delta-rule layer. Requirements: d_model % 64 == 0, ffn % 64 == 0,
 * la_dk == la_dv and la_dk in {64, 128}, fa_head_dim in {64, 128},
 * fa_q_heads % fa_kv_heads == 0, 0 <= conv_width <= 8.
 * conv_width > 0 adds the gated delta rule's short convolution (the snapshot's "convolution
 * history", System1-Omni RFC #114 section 5): each of the q|k|v projection channels of a gated
 * delta-rule layer is convolved causally over rows with its own conv_width taps, then passed
 * through SiLU, before the L2 norms; a sequence continues the last conv_width - 1 input rows of
 * the snapshot it continues (zeros at a sequence start), and a snapshot keeps its own. */
typedef struct {
  int32_t vocab, d_model, n_layers, ffn;
  int32_t la_heads, la_dk, la_dv;               /* gated delta-rule layers             */
  int32_t fa_q_heads, fa_kv_heads, fa_head_dim; /* full-attention layers               */
  const uint8_t* layer_is_full;                 /* [n_layers]                          */
  float rope_theta, rms_eps, l2_eps;            /* e.g. 1e6, 1e-6, 1e-6                */
  int32_t lora_rank;                            /* 0 = no adapter                      */
  float lora_alpha;                             /* delta scale = lora_alpha/lora_rank  */
  int32_t weight_dtype;                         /* S1_F32 or S1_BF16 host arrays       */
  int32_t max_rows;                             /* rows per forward call; 0 -> 32768   */
  int32_t conv_width;                           /* 0 = no short convolution            */
} s1_shape;

/* Host weight arrays, copied at create time (caller keeps ownership).
 * `layer` is the concatenation, layer by layer, of each layer's tensors in this order:
 *   gated delta-rule layer: attn_norm[d], w_q[H*dk,d], w_k[H*dk,d], w_v[H*dv,d],
 *                           w_a[H,d], w_b[H,d], w_o[d,H*dv], mlp_norm[d],
 *                           w_gate[F,d], w_up[F,d], w_down[d,F]            (11 tensors)
 *                           and, when conv_width > 0, conv[2*H*dk + H*dv, conv_width] (12):
 *                           channel c's taps, tap j weighting the input row conv_width-1-j
 *                           rows back (tap conv_width-1 is the current row)
 *   full-attention layer:   attn_norm[d], w_q[Hq*hd,d], w_k[Hkv*hd,d], w_v[Hkv*hd,d],
 *                           w_o[d,Hq*hd], mlp_norm[d], w_gate, w_up, w_down  (9 tensors)
 * lora_a / lora_b: [n_layers*7] pointers, targets in the order q,k,v,o,gate,up,down;
 * A is [rank, in], B is [out, rank]; a NULL pair (or NULL arrays) means no delta. */
typedef struct {
  const void* embed;             /* [vocab, d], tied input/output embedding */
  const void* final_norm;        /* [d] */
  const void* const* layer;
  const void* const* lora_a;
  const void* const* lora_b;
} s1_weights;

/* One question. suffix: token ids in [0, vocab), n_suffix >= 1. option_ids: ids in
 * [0, vocab); choice: n_options >= 1; score: n_options >= 2 (levels in order);
 * noul: exactly 2 ids, {yes, no}. */
typedef struct {
  int32_t type;
  const int32_t* suffix;
  int32_t n_suffix;
  const int32_t* option_ids;
  int32_t n_options;
} s1_question;

/* One result. probs: caller-allocated [n_options]. argmax: most likely option
 * (ties -> lowest index). expected_score: sum_i i*p_i. yes_prob: p[0].
 * answer_confidence: max_i p_i. confidence: 1 - H(p)/ln(n) for choice/score,
 * answer_confidence for noul. entropy_confidence: 1 - H(p)/ln(n) for every type
 * (1 when n == 1). lm_logprobs: NULL, or caller-allocated [n_options] that receives each
 * option token's log-probability under the full vocabulary at the readout row,
 * z_o - log sum_v exp(z_v) over all vocab rows of the tied embedding (System1-Omni RFC #114,
 * section 4 "Readout" and the LM-feature paragraph after its table); renormalising these over
 * the options gives back probs. Requesting it for any question of a call streams the whole
 * embedding once more (blocking calls only). */
typedef struct {
  float* probs;
  int32_t argmax;
  float expected_score;
  float yes_prob;
  float answer_confidence;
  float confidence;
  float entropy_confidence;
  float* lm_logprobs;
} s1_result;

/* Per-question statistics written by the stream-ordered decide (device floats). */
enum { S1_STAT_ARGMAX = 0, S1_STAT_EXPECTED, S1_STAT_YES, S1_STAT_ANSWER_CONF,
       S1_STAT_CONF, S1_STAT_ENTROPY_CONF, S1_STAT_MARGIN, S1_STAT_COUNT = 8 };

/* ---- model ----------------------------------------------------------------------
 * Validates the shape, uploads the weights, merges each LoRA pair as
 * W + (alpha/rank) * B A in fp32 and rounds once to f16 (round to nearest even): every
 * tensor-core operand of the forward pass is f16 (the tensor cores' bf16 rate, three more
 * mantissa bits; a bf16 weight converts to f16 exactly when |w| >= 2^-14, and to within 2^-25
 * below it). The tied embedding is kept as an f16 copy too.
 * Blocking. Errors: INVALID_ARG (shape), UNSUPPORTED, OOM, CUDA. */
int s1_model_create(const s1_shape* shape, const s1_weights* weights, s1_model** out);
void s1_model_destroy(s1_model* m);      /* waits for the model's stream first */

/* Use `stream` (a cudaStream_t, may be NULL = legacy default) for all later work. */
int s1_set_stream(s1_model* m, void* stream);

/* Device-memory hooks used for every later allocation (NULL, NULL restores
 * cudaMalloc / cudaFree). Must be set before s1_model_create. */
int s1_set_allocator(void* (*alloc)(size_t bytes, void* ctx), void (*free_fn)(void* p, void* ctx), void* ctx);

/* ---- prefix --------------------------------------------------------------------------
 * Prefill the state prefix: n_embeds given embedding rows (bf16 [n_embeds, d], host),
 * followed by n_tokens token rows; positions 0 .. n_embeds+n_tokens-1. Returns an
 * immutable snapshot (per-layer gated delta-rule state, fp32 [H, dv, dk], and
 * post-RoPE K/V, f16 [P, Hkv, hd]). Host pointers; blocking.
 * Errors: INVALID_ARG (ids, empty prefix), BUDGET (rows > max_rows), OOM, CUDA. */
int s1_prefill_state(s1_model* m, const int32_t* tokens, int32_t n_tokens,
                     const void* embeds, int32_t n_embeds, s1_state** out);

/* n_req prefixes in one layer sweep (rows packed, one GEMM per projection). */
int s1_prefill_state_batch(s1_model* m, int32_t n_req, const int32_t* const* tokens,
                           const int32_t* n_tokens, const void* const* embeds,
                           const int32_t* n_embeds, s1_state** out);

void s1_state_destroy(s1_state* st);
int s1_state_rows(const s1_state* st);   /* prefix rows P, or -1 for an invalid handle */

/* ---- decisions -------------------------------------------------------------------------
 * Every question continues from the same prefix snapshot (never written); its
 * rows sit at positions P .. P+n_suffix-1. Writes out[j] (probs into out[j].probs)
 * and, if last_hidden != NULL, the last decoder layer's output at the question's
 * last row, before the final norm ([n_q, d] fp32). Host pointers; blocking.
 * Errors: INVALID_HANDLE, INVALID_ARG, BUDGET, OOM, CUDA, DEVICE_TIMEOUT. */
int s1_decide(s1_model* m, const s1_state* st, const s1_question* qs, int32_t n_q,
              s1_result* out, float* last_hidden);

/* Questions of n_req requests, each against its own state, in one layer sweep.
 * last_hidden may be NULL, or an array of n_req pointers (entries may be NULL). */
int s1_decide_batch(s1_model* m, int32_t n_req, const s1_state* const* states,
                    const s1_question* const* qs, const int32_t* n_q,
                    s1_result* const* out, float* const* last_hidden);

/* ---- one sweep: prefix and questions together ---------------------------------------------
 * Same results as s1_prefill_state followed by s1_decide, computed in one pass over the
 * layers: each layer's projections run once over the prefix rows and all suffix rows (the
 * weights are read once per request), the gated delta-rule state pass runs the prefix and
 * then the suffixes from the just-written snapshot, and suffix queries read the prefix K/V
 * the same layer has just cached (System1-Omni RFC #114, section 5: encode the prefix once,
 * then the isolated suffixes, in bounded batches). state_out (may be NULL) receives the
 * prefix snapshot for further s1_decide calls. Host pointers; blocking. */
int s1_prefill_decide(s1_model* m, const int32_t* tokens, int32_t n_tokens, const void* embeds,
                      int32_t n_embeds, const s1_question* qs, int32_t n_q, s1_result* out,
                      float* last_hidden, s1_state** state_out);
/* n_req requests (each a prefix with its questions) in one sweep; last_hidden and states_out
 * may be NULL, or arrays of n_req entries (entries may be NULL for last_hidden). */
int s1_prefill_decide_batch(s1_model* m, int32_t n_req, const int32_t* const* tokens,
                            const int32_t* n_tokens, const void* const* embeds,
                            const int32_t* n_embeds, const s1_question* const* qs,
                            const int32_t* n_q, s1_result* const* out, float* const* last_hidden,
                            s1_state** states_out);

/* ---- stream-ordered variants (device pointers, no host synchronisation) ----------------
 * For callers whose inputs are already in device memory. Host-side metadata
 * (lengths, types, counts) is still passed in host structs; the id arrays they
 * point to are DEVICE pointers and are not range-checked (caller's duty).
 * s1_state_create reserves a state for up to capacity_rows prefix rows;
 * s1_prefill_async (re)fills it. s1_decide_async writes probs (concatenated in
 * question order, [sum n_options] fp32), stats ([n_q, S1_STAT_COUNT] fp32) and
 * optionally last_hidden ([n_q, d] fp32), all device pointers. */
int s1_state_create(s1_model* m, int32_t capacity_rows, s1_state** out);
int s1_prefill_async(s1_model* m, s1_state* st, const int32_t* d_tokens, int32_t n_tokens,
                     const void* d_embeds, int32_t n_embeds);
int s1_decide_async(s1_model* m, const s1_state* st, const s1_question* qs_dev, int32_t n_q,
                    float* d_probs, float* d_stats, float* d_last_hidden);
/* one sweep (as s1_prefill_decide) into a state from s1_state_create; outputs as s1_decide_async */
int s1_prefill_decide_async(s1_model* m, s1_state* st, const int32_t* d_tokens, int32_t n_tokens,
                            const void* d_embeds, int32_t n_embeds, const s1_question* qs_dev,
                            int32_t n_q, float* d_probs, float* d_stats, float* d_last_hidden);

/* one sweep over a batch (as s1_prefill_decide_batch) into n_req states from s1_state_create:
 * request r's prefix is d_embeds[r] (bf16 [n_embeds[r], d], device; the arrays may be NULL) then
 * d_tokens[r] (device ids), its questions qs_dev[r][0 .. n_q[r]) with device id arrays; outputs as
 * s1_decide_async, concatenated over the requests in order. */
int s1_prefill_decide_batch_async(s1_model* m, int32_t n_req, s1_state* const* states,
                                  const int32_t* const* d_tokens, const int32_t* n_tokens,
                                  const void* const* d_embeds, const int32_t* n_embeds,
                                  const s1_question* const* qs_dev, const int32_t* n_q, float* d_probs,
                                  float* d_stats, float* d_last_hidden);

/* CUDA graphs for the stream-ordered calls s1_prefill_async, s1_decide_async,
 * s1_prefill_decide_async and s1_prefill_decide_batch_async (off by default). While enabled, a call whose signature — the
 * function, the state handle, its buffers and capacity (and, for s1_decide_async, its prefix
 * length), every device pointer, size and question type it passes — repeats an earlier call's
 * is captured once into a CUDA graph (its second occurrence) and later occurrences replay that
 * graph with one launch: the ids, embeddings and outputs are
 * read and written through the same device buffers at replay time, so their contents may change
 * between calls while their addresses and sizes may not. Graphs are not used on the legacy
 * default stream, while profiling or a layer trace is on. A graph is dropped when the model's
 * scratch buffers grow, and all are dropped by s1_set_graphs(m, 0) and s1_model_destroy. At
 * most 64 graphs are kept per model; further signatures run without one.
 * Synchronises the model's stream. Errors: INVALID_HANDLE. */
int s1_set_graphs(struct s1_model* m, int enable);
int s1_sync(s1_model* m);   /* waits for the stream; reports device-side timeouts */

/* ---- prefix split (host only) ------------------------------------------------------------
 * For callers that hold one whole token stream per question: the length P of the prefix the
 * streams share, to be prefilled once (System1-Omni RFC #114, implementer's plan comment: the
 * questions' longest common token prefix, cut at least one token before the end of every
 * stream, runs once; the native split may sit at multiples of 64). P is the longest common
 * prefix of the n streams, capped at (shortest length - min_suffix), then rounded down to a
 * multiple of `align` when align > 1 (align = 64 matches the scan's chunk length). Writes P
 * (>= 0) to *prefix_len. Errors: INVALID_ARG (n < 1, a NULL stream, min_suffix < 1, a stream
 * shorter than min_suffix). No device work. */
int s1_split_prefix(const int32_t* const* streams, const int32_t* lens, int32_t n, int32_t min_suffix,
                    int32_t align, int32_t* prefix_len);

const char* s1_last_error(void);
const char* s1_version(void);

#ifdef __cplusplus
}
#endif
#endif /* S1_H_ */
